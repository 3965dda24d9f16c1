"""spd_sparse_decode_attention_static: the decode attention entry point for
callers that cannot allocate device memory when they run attention (inside
stream capture, under a memory plan fixed at start-up, or embedded in a
framework that owns every device allocation).  Its temporaries live in a
library-owned device array; it runs the same kernel as
spd_sparse_decode_attention, so its outputs must be bit-identical to that
entry point's, and within the usual tolerances of the oracle.  This file is
collected last so that a run that stops at the first failure has run every
other test before it."""
import numpy as np
import pytest
import torch

import workloads as W
from harness import TOL_MAX, TOL_MEAN, Pair, tdev
import sparse_paged_decode_logical_gb300 as spd

pytestmark = pytest.mark.gpu
needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")


def _cache(streaming, sink, window, context, token_budget=256):
    cfg = dict(num_q_heads=8, num_kv_heads=4, head_dim=128, dtype="bf16", logical_page=32,
               physical_page=128, num_physical_pages=-(-(context + 64) // 128) * 2,
               max_seqs=2, max_context=context + 64, streaming=streaming, sink=sink,
               window=window, token_budget=token_budget, reuse_interval=4)
    c = spd.SparsePagedKVCache(device="cuda", **cfg)
    g = torch.Generator(device="cuda").manual_seed(7)
    ids = [c.seq_create(), c.seq_create()]
    for s, L in zip(ids, (context, context // 3)):
        k = torch.randn((1, L, 4, 128), generator=g, device="cuda").to(torch.bfloat16)
        v = torch.randn((1, L, 4, 128), generator=g, device="cuda").to(torch.bfloat16)
        c.kv_append([s], k, v)
    return c, ids, g


def _step(c, ids, g):
    q = torch.randn((2, 8, 128), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((2, 4, 128), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((2, 4, 128), generator=g, device="cuda").to(torch.bfloat16)
    c.decode_step(q, k, v, ids)
    return torch.randn((2, 8, 128), generator=g, device="cuda").to(torch.bfloat16)


@needs_gpu
def test_static_scratch_matches_default_entry_point_on_two_calls():
    c, ids, g = _cache([False, True, False, True], sink=16, window=512, context=5000)
    stream = torch.cuda.current_stream().cuda_stream
    for rnd in range(2):
        q = _step(c, ids, g)  # appends a token and (re)selects when due
        ref = torch.empty((2, 8, 128), dtype=torch.float32, device="cuda")
        spd.spd_sparse_decode_attention(c.ctx, q.data_ptr(), ids, ref.data_ptr(), stream)
        outs = []
        for _ in range(2):  # two calls in a row share (and reuse) the array
            got = torch.full((2, 8, 128), float("nan"), dtype=torch.float32, device="cuda")
            spd.spd_sparse_decode_attention_static(c.ctx, q.data_ptr(), ids, got.data_ptr(),
                                                   stream)
            outs.append(got)
        torch.cuda.synchronize()
        c.check_status()
        for got in outs:
            # the same kernel on the same inputs, another scratch base
            assert torch.equal(got, ref), (rnd, float((got - ref).abs().max()))


def _many_sequences():
    # 70 sequences: more than one decode launch holds (64), so one static
    # call runs two launches that reuse the same array one after the other
    lens = [40 + 37 * b for b in range(70)]
    return W.Workload(name="synthetic", index=9, batch=70, Hq=8, Hkv=4, d=128,
                      context=max(lens), ell=16, P=64, dtype="bf16",
                      streaming=[False, True, False, True], sink=8, window=64,
                      token_budget=64, C=4, steps=2, needle="tokens", needle_frac=0.02,
                      lens=lens)


@needs_gpu
def test_static_scratch_over_several_launches_matches_the_oracle():
    wl = _many_sequences()
    pr = Pair(wl)
    pr.step(0)  # append, select and attend on both sides, checked against the oracle
    q_bits, _, _ = W.step_tokens(wl, 1)
    q = tdev(q_bits, "bf16")
    n = wl.batch
    stream = torch.cuda.current_stream().cuda_stream
    ref = torch.empty((n, 8, 128), dtype=torch.float32, device="cuda")
    spd.spd_sparse_decode_attention(pr.cache.ctx, q.data_ptr(), pr.gids, ref.data_ptr(), stream)
    outs = []
    for _ in range(2):
        before = pr.cache.launch_count()
        got = torch.full((n, 8, 128), float("nan"), dtype=torch.float32, device="cuda")
        spd.spd_sparse_decode_attention_static(pr.cache.ctx, q.data_ptr(), pr.gids,
                                               got.data_ptr(), stream)
        assert pr.cache.launch_count() - before >= 2
        outs.append(got)
    torch.cuda.synchronize()
    pr.cache.check_status()
    for got in outs:
        assert torch.equal(got, ref)
    out = outs[-1].cpu().numpy().astype(np.float64)
    for b in range(n):
        # the oracle on the GPU's own selection (ties within the band may differ)
        s = pr.orc.seqs[pr.oids[b]]
        own = {h: s.sel[h] for h in pr.dyn}
        for h in pr.dyn:
            s.sel[h] = np.array(pr.cache.selection(pr.gids[b], h), np.int32)
        want = pr.orc.attend(pr.oids[b], q_bits[b], advance=False)
        for h in pr.dyn:
            s.sel[h] = own[h]
        err = np.abs(out[b] - want)
        assert float(err.max()) <= TOL_MAX and float(err.mean()) <= TOL_MEAN, (b, err.max())


def _wide_streaming_cache(lengths):
    # 33 streaming kv heads with a 131072-token window: a sequence filling the
    # window needs more split items than the 1024 the array holds (each item
    # takes at most 256 tiles of 16 rows)
    W_ = 131072
    cfg = dict(num_q_heads=33, num_kv_heads=33, head_dim=64, dtype="bf16", logical_page=32,
               physical_page=128, num_physical_pages=1, max_seqs=len(lengths),
               max_context=W_ + 64, streaming=[True] * 33, sink=0, window=W_, token_budget=0,
               reuse_interval=4)
    c = spd.SparsePagedKVCache(device="cuda", **cfg)
    g = torch.Generator(device="cuda").manual_seed(11)
    ids = []
    for L in lengths:
        sid = c.seq_create()
        k = torch.randn((1, L, 33, 64), generator=g, device="cuda").to(torch.bfloat16)
        v = torch.randn((1, L, 33, 64), generator=g, device="cuda").to(torch.bfloat16)
        c.kv_append([sid], k, v)
        del k, v
        ids.append(sid)
    q = torch.randn((len(lengths), 33, 64), generator=g, device="cuda").to(torch.bfloat16)
    return c, ids, q


@needs_gpu
def test_static_scratch_rejects_work_beyond_its_capacity():
    c, ids, q = _wide_streaming_cache([131072 + 16])
    before = c.seq_info(ids[0])["step_counter"]
    out = torch.empty((1, 33, 64), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    with pytest.raises(spd.SpdError) as e:
        spd.spd_sparse_decode_attention_static(c.ctx, q.data_ptr(), ids, out.data_ptr(), stream)
    assert e.value.name == "SPD_ERR_CAPACITY"
    assert c.seq_info(ids[0])["step_counter"] == before
    spd.spd_sparse_decode_attention(c.ctx, q.data_ptr(), ids, out.data_ptr(), stream)
    torch.cuda.synchronize()
    c.check_status()
    assert torch.isfinite(out).all()


@needs_gpu
def test_static_scratch_refuses_before_enqueuing_anything():
    # the first sequence fits on its own, the second does not: the whole call
    # is refused before the first sequence's launch, so its rows of `out` are
    # never written and no step counter moves
    c, ids, q = _wide_streaming_cache([2000, 131072 + 16])
    before = [c.seq_info(s)["step_counter"] for s in ids]
    out = torch.full((2, 33, 64), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    with pytest.raises(spd.SpdError) as e:
        spd.spd_sparse_decode_attention_static(c.ctx, q.data_ptr(), ids, out.data_ptr(), stream)
    assert e.value.name == "SPD_ERR_CAPACITY"
    torch.cuda.synchronize()
    c.check_status()
    assert torch.isnan(out).all()
    assert [c.seq_info(s)["step_counter"] for s in ids] == before
