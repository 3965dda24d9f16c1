"""A multi-layer decode step: layers with different head-type assignments
(all-streaming, all-dynamic and mixed; LServe write-up, section 2.1: static
sparsity turns some heads -- up to whole layers -- into streaming heads), each
layer its own context, every layer's decode step of several steps captured
into one CUDA graph and replayed once, with early KV staging across layers.
Checked against the oracle layer by layer and step by step."""
import numpy as np
import pytest
import torch

import workloads as W
from harness import TOL_MAX, TOL_MEAN, Pair, tdev

pytestmark = pytest.mark.gpu

needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")

MASKS = [[False, True, False, True],   # mixed
         [True, True, True, True],     # an all-streaming layer
         [False, False, False, False], # an all-dynamic layer
         [True, False, False, True]]   # mixed, the other way round


@needs_gpu
def test_layers_with_different_head_types_in_one_graph():
    wl = W.Workload(name="synthetic", index=11, batch=2, Hq=8, Hkv=4, d=128, context=900,
                    ell=16, P=64, dtype="bf16", streaming=MASKS[0], sink=8, window=40,
                    token_budget=128, C=3, steps=6, needle="tokens", needle_frac=0.02,
                    lens=[900, 333])
    pairs = [Pair(wl, layer=l, cfg_overrides={"streaming": m}) for l, m in enumerate(MASKS)]
    for pr in pairs:
        pr.cache.set_early_kv_staging(True)
    stream = torch.cuda.Stream()
    # step 0 eagerly (the first call binds each context to the device)
    with torch.cuda.stream(stream):
        for pr in pairs:
            pr.step(0)
    steps = list(range(1, wl.steps))
    toks = {(s, l): W.step_tokens(wl, s, l) for s in steps for l in range(len(pairs))}
    dev = {key: tuple(tdev(x, wl.dtype) for x in val) for key, val in toks.items()}
    outs = {key: torch.empty((wl.batch, wl.Hq, wl.d), dtype=torch.float32, device="cuda")
            for key in toks}
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for s in steps:
            for l, pr in enumerate(pairs):
                q, k, v = dev[s, l]
                pr.cache.decode_step(q, k, v, pr.gids, out=outs[s, l])
    g.replay()
    torch.cuda.synchronize()
    for pr in pairs:
        pr.cache.check_status()

    last_q = {}
    for s in steps:
        for l, pr in enumerate(pairs):
            q, k, v = toks[s, l]
            out = outs[s, l].cpu().numpy().astype(np.float64)
            for b in range(wl.batch):
                oid = pr.oids[b]
                pr.orc.append(oid, k[b][None], v[b][None])
                if pr.orc.select(oid, q[b]):
                    last_q[l, b] = q[b]
                ref = pr.orc.attend(oid, q[b])
                err = np.abs(out[b] - ref)
                assert np.isfinite(out[b]).all()
                assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN, (s, l, b, err.max())
    for l, pr in enumerate(pairs):
        pr.check_layout()
        for b in range(wl.batch):
            if pr.dyn:
                pr.check_selection(b, last_q[l, b])
