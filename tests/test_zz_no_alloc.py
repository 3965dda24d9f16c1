"""spd_sparse_decode_attention_static: the decode attention entry point for
callers that cannot allocate device memory when they run attention (inside
stream capture, under a memory plan fixed at start-up, or embedded in a
framework that owns every device allocation).  Its temporaries live in a
library-owned device array; it must give the same outputs as
spd_sparse_decode_attention.  This file is collected last so that a run that
stops at the first failure has run every other test before it."""
import pytest
import torch

import sparse_paged_decode_logical_gb300 as spd

pytestmark = pytest.mark.gpu
needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")

TOL_MAX, TOL_MEAN = 2e-3, 2e-4


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


def _close(a, b):
    d = (a - b).abs()
    return float(d.max()) <= TOL_MAX and float(d.mean()) <= TOL_MEAN


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
            assert torch.isfinite(got).all()
            assert _close(got, ref), (rnd, float((got - ref).abs().max()))


@needs_gpu
def test_static_scratch_rejects_work_beyond_its_capacity():
    # 33 streaming kv heads with a 131072-token window: one sequence needs
    # more split items than the 1024 the array holds (each CTA takes at most
    # 256 tiles of 16 rows), so the call is refused before any launch and the
    # sequence's step counter does not move; the default entry point runs it
    W_ = 131072
    cfg = dict(num_q_heads=33, num_kv_heads=33, head_dim=64, dtype="bf16", logical_page=32,
               physical_page=128, num_physical_pages=1, max_seqs=1, max_context=W_ + 64,
               streaming=[True] * 33, sink=0, window=W_, token_budget=0, reuse_interval=4)
    c = spd.SparsePagedKVCache(device="cuda", **cfg)
    sid = c.seq_create()
    g = torch.Generator(device="cuda").manual_seed(11)
    k = torch.randn((1, W_ + 16, 33, 64), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((1, W_ + 16, 33, 64), generator=g, device="cuda").to(torch.bfloat16)
    c.kv_append([sid], k, v)
    del k, v
    q = torch.randn((1, 33, 64), generator=g, device="cuda").to(torch.bfloat16)
    before = c.seq_info(sid)["step_counter"]
    out = torch.empty((1, 33, 64), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    with pytest.raises(spd.SpdError) as e:
        spd.spd_sparse_decode_attention_static(c.ctx, q.data_ptr(), [sid], out.data_ptr(),
                                               stream)
    assert e.value.name == "SPD_ERR_CAPACITY"
    assert c.seq_info(sid)["step_counter"] == before
    spd.spd_sparse_decode_attention(c.ctx, q.data_ptr(), [sid], out.data_ptr(), stream)
    torch.cuda.synchronize()
    c.check_status()
    assert torch.isfinite(out).all()
