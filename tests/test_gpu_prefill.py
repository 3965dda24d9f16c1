"""GPU parity of the prefill-side block-sparse attention ("LServe long-sequence
LLM serving system", section 3.1) against the CPU oracle, through the C ABI.

Block selection: the GPU's lists equal the oracle's, except blocks whose
oracle score lies within 1e-4 of the row's largest score magnitude of the
cut (the GPU pools then projects in fp32, the oracle projects then pools in
fp64).  Attention: the oracle run on the GPU's own lists, max-abs <= 2e-3
and mean-abs <= 2e-4 (the decode tolerances)."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from harness import TOL_MAX, TOL_MEAN, tdev
import sparse_paged_decode_logical_gb300 as spd

pytestmark = pytest.mark.gpu

needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
BLK = 64
BAND = 1e-4


def _inputs(seed, L, Hq, Hkv, d, r, dtype):
    rg = np.random.default_rng([20260, 77, seed])
    Q = W.to_bits(rg.standard_normal((L, Hq, d)).astype(np.float32), dtype)
    K = W.to_bits(rg.standard_normal((L, Hkv, d)).astype(np.float32), dtype)
    V = W.to_bits(rg.standard_normal((L, Hkv, d)).astype(np.float32), dtype)
    # a planted key block that the low-rank scores favour for some heads
    Wq = (rg.standard_normal((Hkv, d, r)) / np.sqrt(d)).astype(np.float32)
    Wk = (rg.standard_normal((Hkv, d, r)) / np.sqrt(d)).astype(np.float32)
    return Q, K, V, Wq, Wk


def _check(L, Hq, Hkv, d, r, dtype, budget, dense_below, seed):
    Q, K, V, Wq, Wk = _inputs(seed, L, Hq, Hkv, d, r, dtype)
    out, blocks = spd.prefill_block_sparse_attention(
        tdev(Q, dtype), tdev(K, dtype), tdev(V, dtype), torch.from_numpy(Wq).cuda(),
        torch.from_numpy(Wk).cuda(), block=BLK, token_budget=budget, dense_below=dense_below)
    torch.cuda.synchronize()
    out = out.cpu().numpy().astype(np.float64)
    blocks = blocks.cpu().numpy()
    G = Hq // Hkv
    nb = -(-L // BLK)
    for hk in range(Hkv):
        Qh = np.ascontiguousarray(Q[:, hk * G:(hk + 1) * G].transpose(1, 0, 2))
        S = oracle.prefill_block_scores(Qh, K[:, hk], dtype, Wq[hk], Wk[hk], BLK)
        own = oracle.prefill_select(S, BLK, L, budget, dense_below)
        gpu = []
        for b in range(nb):
            row = blocks[hk, b]
            g = row[row >= 0]
            assert np.all(np.diff(g) > 0) and g[-1] == b, (hk, b, g)
            assert np.all(row[len(g):] == -1)
            if not np.array_equal(g, own[b]):
                assert len(g) == len(own[b]), (hk, b)
                cand = [i for i in own[b] if i != b]
                cut = S[b, cand].min()
                tol = BAND * max(np.abs(S[b, :b]).max(), 1e-30)
                diff = np.setxor1d(g, own[b])
                assert np.all(np.abs(S[b, diff] - cut) <= tol), (hk, b, diff, S[b, diff], cut)
            gpu.append(g.astype(np.int32))
        ref = oracle.prefill_attention(Qh, K[:, hk], V[:, hk], dtype, gpu, BLK)  # [G][L][d]
        got = out[:, hk * G:(hk + 1) * G].transpose(1, 0, 2)
        err = np.abs(got - ref)
        assert np.isfinite(got).all()
        assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN, (hk, err.max(), err.mean())
    return blocks


@needs_gpu
def test_prefill_dense_below_the_threshold():
    # 300 tokens: 5 blocks, the last partial; every causal block attended
    blocks = _check(300, 4, 2, 128, 16, "bf16", budget=128, dense_below=32768, seed=1)
    assert blocks.shape == (2, 5, 5)


@needs_gpu
@pytest.mark.parametrize("case", [
    dict(L=1000, Hq=8, Hkv=2, d=128, r=16, dtype="bf16", budget=256, seed=2),
    dict(L=777, Hq=2, Hkv=2, d=64, r=8, dtype="f16", budget=128, seed=3),
    dict(L=500, Hq=8, Hkv=1, d=128, r=16, dtype="bf16", budget=64, seed=4),
    dict(L=2048, Hq=4, Hkv=1, d=128, r=16, dtype="f16", budget=512, seed=5),
    dict(L=1500, Hq=16, Hkv=2, d=64, r=8, dtype="bf16", budget=384, seed=9),
    dict(L=1100, Hq=8, Hkv=4, d=64, r=8, dtype="f16", budget=256, seed=10),
])
def test_prefill_sparse_blocks(case):
    c = dict(case)
    _check(c.pop("L"), c.pop("Hq"), c.pop("Hkv"), c.pop("d"), c.pop("r"), c.pop("dtype"),
           c.pop("budget"), dense_below=0, seed=c.pop("seed"))


@needs_gpu
@pytest.mark.parametrize("case", [
    dict(L=1, Hq=4, Hkv=2, d=128, r=16, dtype="bf16", budget=64, dense_below=0, seed=6),
    dict(L=64, Hq=2, Hkv=1, d=64, r=8, dtype="f16", budget=64, dense_below=0, seed=7),
    dict(L=320, Hq=4, Hkv=4, d=128, r=16, dtype="bf16", budget=10 ** 6, dense_below=0, seed=8),
])
def test_prefill_edges(case):
    # one token; exactly one full block; a budget above the prompt (every block kept)
    c = dict(case)
    _check(c.pop("L"), c.pop("Hq"), c.pop("Hkv"), c.pop("d"), c.pop("r"), c.pop("dtype"),
           c.pop("budget"), c.pop("dense_below"), seed=c.pop("seed"))


def _check_full(L, Hq, Hkv, d, r, dtype, budget, dense_below, seed, sample):
    """A prompt at the measured size: every block list of every kv head against
    the oracle's selection (same band as above), and attention for the query
    blocks in `sample` (first, last, a few between), each query token against
    the oracle's softmax attention over the keys s <= t of its query block's
    GPU-chosen blocks -- the per-token definition the prefill attention of the
    oracle is written from, evaluated only where sampled to keep the CPU side
    affordable."""
    Q, K, V, Wq, Wk = _inputs(seed, L, Hq, Hkv, d, r, dtype)
    out, blocks = spd.prefill_block_sparse_attention(
        tdev(Q, dtype), tdev(K, dtype), tdev(V, dtype), torch.from_numpy(Wq).cuda(),
        torch.from_numpy(Wk).cuda(), block=BLK, token_budget=budget, dense_below=dense_below)
    torch.cuda.synchronize()
    blocks = blocks.cpu().numpy()
    G = Hq // Hkv
    nb = -(-L // BLK)
    dense = L < dense_below
    kept = nb if dense else max(1, budget // BLK)
    assert blocks.shape == (Hkv, nb, kept)
    worst = 0.0
    for hk in range(Hkv):
        Qh = np.ascontiguousarray(Q[:, hk * G:(hk + 1) * G].transpose(1, 0, 2))
        S = oracle.prefill_block_scores(Qh, K[:, hk], dtype, Wq[hk], Wk[hk], BLK)
        own = oracle.prefill_select(S, BLK, L, budget, dense_below)
        lists = []
        for b in range(nb):
            row = blocks[hk, b]
            g = row[row >= 0]
            assert np.all(np.diff(g) > 0) and g[-1] == b, (hk, b)
            assert len(g) == min(b + 1, kept), (hk, b, len(g))
            if not np.array_equal(g, own[b]):
                assert not dense and len(g) == len(own[b]), (hk, b)
                cand = [i for i in own[b] if i != b]
                cut = S[b, cand].min()
                tol = BAND * max(np.abs(S[b, :b]).max(), 1e-30)
                diff = np.setxor1d(g, own[b])
                assert np.all(np.abs(S[b, diff] - cut) <= tol), (hk, b, diff, S[b, diff], cut)
            lists.append(g)
        for b in sample:
            g = lists[b]
            keys = np.concatenate([np.arange(c * BLK, min((c + 1) * BLK, L)) for c in g])
            # the chosen rows only, in ascending position (the same rows and order)
            Ks = np.ascontiguousarray(K[keys, hk])
            Vs = np.ascontiguousarray(V[keys, hk])
            ts = list(range(b * BLK, min((b + 1) * BLK, L)))
            # one oracle call per query token, on the host's cores (the calls
            # release the interpreter lock)
            with ThreadPoolExecutor(oracle.cpu_threads()) as ex:
                refs = list(ex.map(lambda t: oracle.attention(
                    Q[t, hk * G:(hk + 1) * G], Ks, Vs, dtype, np.nonzero(keys <= t)[0]), ts))
            got_b = out[ts[0]:ts[-1] + 1, hk * G:(hk + 1) * G].cpu().numpy().astype(np.float64)
            for x, t in enumerate(ts):
                err = np.abs(got_b[x] - refs[x])
                assert np.isfinite(got_b[x]).all()
                assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN, (hk, b, t, err.max())
                worst = max(worst, float(err.max()))
    return worst


@needs_gpu
def test_prefill_full_size_sparse_across_the_dense_threshold():
    # 32868 tokens: 514 blocks (the last partial), at the 32K threshold, so the
    # sparse rule applies; budget 4096 = 64 kept blocks per query block, which
    # every block from the 64th on has to choose from its earlier ones
    L = 32768 + 100
    _check_full(L, 8, 2, 128, 16, "bf16", budget=4096, dense_below=32768, seed=11,
                sample=[0, 1, 63, 64, 257, 511, 513])


@needs_gpu
def test_prefill_full_size_one_token_below_the_threshold_is_dense():
    # 32767 tokens: one below the threshold, every causal block attended
    _check_full(32767, 4, 1, 128, 16, "f16", budget=4096, dense_below=32768, seed=12,
                sample=[0, 255, 511])


@needs_gpu
def test_prefill_full_size_eight_heads_per_kv_head_fp16():
    # 40,000 tokens (625 blocks, the last partial), 8 query heads per kv head
    # (two CTAs per query block and kv head on the tensor-core path), fp16
    # (the rounded 16-bit high part of P), budget 2048 = 32 kept blocks
    _check_full(40000, 16, 2, 128, 16, "f16", budget=2048, dense_below=32768, seed=13,
                sample=[0, 31, 32, 400, 624])
