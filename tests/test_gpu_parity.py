"""GPU parity: the CUDA library, called through the C ABI, against the CPU
oracle on the same seeded inputs.  Element by element on every output."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from harness import Pair, tdev
import sparse_paged_decode_logical_gb300 as spd

pytestmark = pytest.mark.gpu

needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")


def run(wl, steps=None, layout_every=4, **kw):
    pr = Pair(wl, **kw)
    pr.check_layout()
    for s in range(wl.steps if steps is None else steps):
        pr.step(s, check_layout=(s % layout_every == layout_every - 1))
    pr.check_layout()
    return pr


@needs_gpu
def test_tiny_workload():
    # 1 sequence, GQA 4/2, d 64, 4096 tokens, fp16; kv 0 dynamic (budget 512),
    # kv 1 streaming (16 + 256); 8 steps with C = 4
    pr = run(W.workload("tiny"), layout_every=1)
    sel_steps = [r["step"] for r in pr.records if r["selected"]]
    assert sel_steps == [0, 4]


@needs_gpu
def test_selection_reused_between_selection_steps():
    wl = W.workload("tiny", steps=9, context=1000)
    pr = Pair(wl)
    sels = []
    for s in range(wl.steps):
        pr.step(s)
        sels.append(pr.cache.selection(pr.gids[0], 0))
    for s in range(wl.steps):
        if s % 4:
            assert sels[s] == sels[s - s % 4]


@needs_gpu
@pytest.mark.parametrize("name", ["llama3_8b_b4_32k", "llama3_8b_b1_128k"])
def test_full_size_workloads(name):
    wl = W.workload(name)
    run(wl, steps=min(wl.steps, 9), layout_every=8)


@needs_gpu
def test_llama2_mha_reduced_context():
    # MHA 32/32 with logical page 64; the 256K context is exercised by the
    # benchmark-shape test below, here 64K keeps the oracle quick
    run(W.workload("llama2_7b_mha_256k", context=65536), steps=6, layout_every=3)


@needs_gpu
def test_continuous_batch_mixed_lengths():
    # 16 sequences, log-uniform lengths (scaled down 8x from [8K, 128K]),
    # shared pool in random order, budget min(4096, L/32)
    wl = W.workload("cont_batch_16", log_uniform_lens=(1024, 16384))
    pr = run(wl, steps=9, layout_every=4)
    assert len(set(pr.lens)) > 10


def synth(**kw):
    base = dict(name="synthetic", index=9, batch=2, Hq=8, Hkv=4, d=128, context=700,
                ell=16, P=64, dtype="bf16", streaming=[False, True, False, True],
                sink=8, window=40, token_budget=128, C=3, steps=7, needle="tokens",
                needle_frac=0.02)
    base.update(kw)
    return W.Workload(**base)


SHAPES = [
    dict(),
    dict(dtype="f16", d=64, Hq=16, Hkv=2, streaming=[False, True], ell=32, P=128),
    dict(Hq=4, Hkv=4, streaming=[False] * 4, ell=64, P=256, token_budget=0, context=9000),
    dict(Hq=32, Hkv=4, streaming=[True, False, False, True], sink=0, window=1),
    dict(streaming=[True] * 4, context=50, window=30, sink=4),
    dict(streaming=[False] * 4, token_budget=10 ** 6, context=333),
    dict(token_budget=16, context=301),
    dict(context=1, steps=5, batch=3),
    dict(context=63, steps=4, C=1, lens=[63, 64, 65]),
    dict(batch=5, lens=[1, 17, 64, 640, 1000], steps=6, permute_pages=True),
]


@needs_gpu
@pytest.mark.parametrize("shape", range(len(SHAPES)))
def test_synthetic_shapes_and_edges(shape):
    kw = SHAPES[shape]
    if "lens" in kw:
        kw = dict(kw, batch=len(kw["lens"]))
    run(synth(**kw), layout_every=2)


@needs_gpu
def test_physical_page_permutation_leaves_outputs_unchanged():
    # the pool order changes only where pages live, never what is computed:
    # outputs are bit-identical under a random permutation of physical pages
    wl = synth(context=900, steps=5, batch=2)
    outs, tables = [], []
    for seed in (0, 77):
        pr = Pair(wl, cfg_overrides=dict(free_list_seed=seed, num_physical_pages=64))
        tables.append(pr.cache.page_table(pr.gids[0]))
        res = []
        for s in range(wl.steps):
            q, k, v = W.step_tokens(wl, s)
            res.append(pr.cache.decode_step(tdev(q, wl.dtype), tdev(k, wl.dtype),
                                            tdev(v, wl.dtype), pr.gids).cpu())
        outs.append(torch.stack(res))
    assert tables[0] != tables[1]
    assert torch.equal(outs[0], outs[1])


@needs_gpu
def test_sequence_free_and_page_reuse():
    wl = synth(batch=2, context=500, steps=3)
    pr = Pair(wl, cfg_overrides=dict(num_physical_pages=24))
    for s in range(2):
        pr.step(s)
    free0 = pr.cache.free_pages()
    pr.cache.seq_free(pr.gids[0])
    pr.orc.free_seq(pr.oids[0])
    assert pr.cache.free_pages() > free0
    # a new sequence takes the freed pages; old contents must not leak
    pr.gids[0] = pr.cache.seq_create()
    pr.oids[0] = pr.orc.new_seq()
    K, V = W.context(wl, 0, 300, layer=5)
    pr.append_seq(0, K, V)
    pr.check_layout()
    pr.step(2)
    pr.check_layout()


@needs_gpu
def test_fused_step_equals_separate_calls():
    # spd_decode_step (append fused into the decode kernel) and the three
    # entry points called one by one must give bit-identical outputs, pools
    # and metadata
    wl = synth(batch=3, lens=[37, 300, 1000], steps=6, ell=32, P=128)
    a = Pair(wl)
    b = Pair(wl)
    for s in range(wl.steps):
        q, k, v = W.step_tokens(wl, s)
        qd, kd, vd = tdev(q, wl.dtype), tdev(k, wl.dtype), tdev(v, wl.dtype)
        oa = a.cache.decode_step(qd, kd, vd, a.gids)
        b.cache.kv_append(b.gids, kd[:, None].contiguous(), vd[:, None].contiguous())
        b.cache.select_pages(qd, b.gids)
        ob = b.cache.sparse_decode_attention(qd, b.gids)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob), s
    # both sides' pools, rings and metadata hold what the oracle holds; the
    # oracle state was never advanced here, so feed it the same tokens first
    for pr in (a, b):
        for s in range(wl.steps):
            q, k, v = W.step_tokens(wl, s)
            for i in range(wl.batch):
                pr.orc.append(pr.oids[i], k[i][None], v[i][None])
        pr.check_layout()


@needs_gpu
def test_launch_counts():
    wl = synth(batch=1, context=500, steps=1)
    pr = Pair(wl)
    n0 = pr.cache.launch_count()
    q, k, v = W.step_tokens(wl, 0)
    pr.cache.decode_step(tdev(q, wl.dtype), tdev(k, wl.dtype), tdev(v, wl.dtype), pr.gids)
    # a selection step: fused score+top-k, then the fused append+decode kernel
    # (plus a page-table write when the token opens a physical page)
    assert pr.cache.launch_count() - n0 in (2, 3)


@needs_gpu
def test_early_kv_staging_interleaved_contexts_bit_identical():
    # three contexts stepped round-robin on one stream (like consecutive
    # layers): with early staging each decode kernel loads its tiles while the
    # previous context's kernel finishes; outputs must equal the default path
    wl = synth(batch=2, lens=[700, 1500], steps=9, ell=32, P=128)
    res = []
    for early in (False, True):
        prs = [Pair(wl, layer=layer) for layer in range(3)]
        for pr in prs:
            pr.cache.set_early_kv_staging(early)
        outs = []
        for s in range(wl.steps):
            for layer, pr in enumerate(prs):
                q, k, v = W.step_tokens(wl, s, layer)
                outs.append(pr.cache.decode_step(tdev(q, wl.dtype), tdev(k, wl.dtype),
                                                 tdev(v, wl.dtype), pr.gids))
        torch.cuda.synchronize()
        for pr in prs:
            pr.cache.check_status()
        res.append(torch.stack([o.cpu() for o in outs]))
    assert torch.equal(res[0], res[1])


@needs_gpu
def test_llama2_mha_full_256k():
    # Llama-2-7B attention (MHA 32/32, d 128, fp16) at 262144 tokens, logical
    # page 64: the full-size workload, two selections (steps 0 and 4)
    run(W.workload("llama2_7b_mha_256k"), steps=5, layout_every=5)


@needs_gpu
def test_continuous_batch_full_lengths():
    # 16 sequences at their seeded log-uniform lengths in [8K, 128K], shared
    # permuted pool, budget min(4096, L/32): full-size, first selection plus
    # one reuse step
    wl = W.workload("cont_batch_16")
    pr = run(wl, steps=2, layout_every=2)
    assert max(pr.lens) > 65536 and min(pr.lens) < 16384


# ---- selection fallbacks ------------------------------------------------------
# A fused decode step has the decode kernel select the pages from a bounded
# candidate list; these cases take the other routes, which must agree with the
# oracle just the same.

@needs_gpu
def test_more_due_sequences_than_one_selection_launch():
    # 70 sequences due in one step: more than one selection launch holds, so
    # the selection kernel selects (in two launches) instead of the decode kernel
    wl = synth(batch=70, context=300, ell=16, P=64, token_budget=64, steps=3,
               streaming=[False, True, False, True])
    run(wl, layout_every=3)


@needs_gpu
def test_tied_scores_keep_the_lowest_pages():
    # constant keys: every page has the same bounds and every score ties, so
    # all 1,250 candidates reach the bound (more than the bounded list holds)
    # and the selection is the lowest pages plus the newest one
    wl = synth(batch=1, context=20000, ell=16, P=256, streaming=[False] * 4,
               token_budget=1024, steps=3, needle="none", needle_frac=0.0)
    pr = Pair(wl, prefill=False)
    rng = np.random.default_rng(5)
    K = np.full((wl.context, wl.Hkv, wl.d), 0.5, np.float32)
    V = rng.standard_normal((wl.context, wl.Hkv, wl.d), dtype=np.float32)
    pr.append_seq(0, W.to_bits(K, wl.dtype), W.to_bits(V, wl.dtype))
    for s in range(wl.steps):
        pr.step(s)
    k_sel = oracle.budget_pages(wl.context + 1, wl.token_budget, wl.ell)
    for h in pr.dyn:
        sel = np.array(pr.cache.selection(pr.gids[0], h))
        assert np.array_equal(sel[:-1], np.arange(k_sel - 1)), sel[:8]
    pr.check_layout()


@needs_gpu
def test_more_candidate_pages_than_a_fused_step_holds():
    # 8,749 candidate pages (140,000 tokens of 16-token pages): beyond what a
    # fused step keeps in shared memory, so the selection kernel's global-memory
    # top-k selects
    wl = synth(batch=1, Hq=2, Hkv=1, d=64, streaming=[False], context=140000, ell=16,
               P=256, token_budget=4096, steps=2)
    run(wl, layout_every=2)


# ---- softmax statistics export ------------------------------------------------
# row max: fp32 logits of exact 16-bit products (<= 128 terms): relative error
# <= 128 * 2^-24 < 1e-5 of the logit scale, so 1e-4 absolute per unit of |m|;
# row sum: fp32 exponentials summed over <= 8K terms in a tree, 1e-3 relative.
TOL_STAT_M, TOL_STAT_L = 1e-4, 1e-3


def _check_stats(pr, q):
    out, rm, rs = pr.cache.sparse_decode_attention_stats(tdev(q, pr.dt), pr.gids)
    pr.cache.check_status()
    out, rm, rs = (t.cpu().numpy().astype(np.float64) for t in (out, rm, rs))
    for b in range(pr.wl.batch):
        oid, s = pr.oids[b], pr.orc.seqs[pr.oids[b]]
        own = {h: s.sel[h] for h in pr.dyn}
        for h in pr.dyn:  # the oracle on the GPU's own selection
            s.sel[h] = np.array(pr.cache.selection(pr.gids[b], h), np.int32)
        m_o, l_o = pr.orc.softmax_stats(oid, q[b])
        ref = pr.orc.attend(oid, q[b])
        for h in pr.dyn:
            s.sel[h] = own[h]
        assert np.all(np.abs(rm[b] - m_o) <= TOL_STAT_M * np.maximum(1.0, np.abs(m_o))), b
        assert np.all(np.abs(rs[b] - l_o) <= TOL_STAT_L * l_o), b
        err = np.abs(out[b] - ref)
        assert err.max() <= 2e-3 and err.mean() <= 2e-4, b


@needs_gpu
@pytest.mark.parametrize("which", ["synthetic", "llama3_8b_b4_32k"])
def test_softmax_statistics_export(which):
    wl = synth(batch=3, lens=[40, 700, 1500], steps=3) if which == "synthetic" \
        else W.workload(which)
    pr = Pair(wl)
    for s in range(2):
        pr.step(s)
    q, _, _ = W.step_tokens(wl, 2)
    _check_stats(pr, q)


# ---- per-page attention mass ---------------------------------------------------
# a page's mass is a sum of fp32 exp2 weights over its <= 64 rows (logits of
# exact 16-bit products, relative error < 1e-5) over the fp32 row sum: well
# inside 1e-4 absolute for a quantity in [0, 1]
TOL_MASS = 1e-4


def _check_page_mass(pr, q, max_pages=None):
    out, rm, rs, pages, mass = pr.cache.sparse_decode_attention_page_mass(
        tdev(q, pr.dt), pr.gids, max_pages=max_pages)
    pr.cache.check_status()
    out, rm, rs, mass = (t.cpu().numpy().astype(np.float64) for t in (out, rm, rs, mass))
    pages = pages.cpu().numpy()
    assert pages.shape[:2] == (pr.wl.batch, len(pr.dyn))
    for b in range(pr.wl.batch):
        oid, s = pr.oids[b], pr.orc.seqs[pr.oids[b]]
        own = {h: s.sel[h] for h in pr.dyn}
        for h in pr.dyn:  # the oracle on the GPU's own selection
            s.sel[h] = np.array(pr.cache.selection(pr.gids[b], h), np.int32)
        ref_mass = pr.orc.page_mass(oid, q[b])
        m_o, l_o = pr.orc.softmax_stats(oid, q[b])
        ref = pr.orc.attend(oid, q[b])
        for h in pr.dyn:
            s.sel[h] = own[h]
        for hd, h in enumerate(pr.dyn):
            pg, ms = ref_mass[h]
            n = pg.size
            assert np.array_equal(pages[b, hd, :n], pg), (b, h)
            assert np.all(pages[b, hd, n:] == -1), (b, h)
            err = np.abs(mass[b, hd, :, :n] - ms)
            assert err.max() <= TOL_MASS, (b, h, err.max())
            assert np.all(mass[b, hd, :, n:] == 0.0), (b, h)
            assert np.allclose(mass[b, hd].sum(-1), 1.0, rtol=0, atol=TOL_MASS), (b, h)
        assert np.all(np.abs(rm[b] - m_o) <= TOL_STAT_M * np.maximum(1.0, np.abs(m_o))), b
        assert np.all(np.abs(rs[b] - l_o) <= TOL_STAT_L * l_o), b
        err = np.abs(out[b] - ref)
        assert err.max() <= 2e-3 and err.mean() <= 2e-4, b


PAGE_MASS_CASES = {
    # ragged lengths, 8 kept pages of 16 tokens, streaming heads beside
    "synthetic": lambda: synth(batch=3, lens=[40, 700, 1500], steps=3),
    # 64-token pages: 4 tiles a page, the newest one partial
    "ell64": lambda: synth(Hq=4, Hkv=4, streaming=[False] * 4, ell=64, P=256, token_budget=0,
                           context=9000, batch=1, steps=3),
    # 1024 kept pages on one dynamic head: the unit spans several clusters
    "many_clusters": lambda: synth(Hq=4, Hkv=2, streaming=[False, True], context=30000,
                                   token_budget=16384, batch=1, steps=3),
    "llama3_8b_b4_32k": lambda: W.workload("llama3_8b_b4_32k"),
}


@needs_gpu
@pytest.mark.parametrize("which", list(PAGE_MASS_CASES))
def test_page_mass_export(which):
    wl = PAGE_MASS_CASES[which]()
    pr = Pair(wl)
    for s in range(2):
        pr.step(s)
    q, _, _ = W.step_tokens(wl, 2)
    _check_page_mass(pr, q)
    # a roomier output: the extra entries are padding
    q, _, _ = W.step_tokens(wl, 3)
    _check_page_mass(pr, q, max_pages=max(pr.cache.attended_page_count(g) for g in pr.gids) + 5)


@needs_gpu
def test_page_mass_capacity_is_checked_before_any_work():
    wl = synth(batch=2, lens=[700, 1500], steps=3)
    pr = Pair(wl)
    pr.step(0)
    q, _, _ = W.step_tokens(wl, 1)
    before = [pr.cache.seq_info(g) for g in pr.gids]
    with pytest.raises(spd.SpdError) as e:
        pr.cache.sparse_decode_attention_page_mass(tdev(q, pr.dt), pr.gids, max_pages=3)
    assert e.value.name == "SPD_ERR_CAPACITY"
    assert [pr.cache.seq_info(g) for g in pr.gids] == before
    _check_page_mass(pr, q)


# ---- fp8 (E4M3) KV storage -------------------------------------------------------
# Codes and metadata bit-exact against the oracle's quantisation (fp32 division,
# round to nearest even, saturation); attention against the oracle over the
# dequantised values (code * scale), same tolerances.  One key scale is small
# enough that large keys saturate at 448.
FP8 = dict(kv_fp8=True, k_scale=[0.05, 0.004, 1.0, 0.5], v_scale=[0.1, 2.0, 0.03, 1.0])
FP8_SHAPES = [
    dict(),
    dict(dtype="f16"),
    dict(Hq=4, Hkv=4, streaming=[False] * 4, ell=64, P=256, token_budget=0, context=9000),
    dict(Hq=32, Hkv=4, streaming=[True, False, False, True], sink=0, window=1),
    dict(context=1, steps=5, batch=3),
    dict(batch=5, lens=[1, 17, 64, 640, 1000], steps=6, permute_pages=True),
]


def _fp8_cfg(wl):
    return {k: (v[:wl.Hkv] if isinstance(v, list) else v) for k, v in FP8.items()}


@needs_gpu
@pytest.mark.parametrize("shape", range(len(FP8_SHAPES)))
def test_fp8_kv_shapes_and_edges(shape):
    kw = FP8_SHAPES[shape]
    if "lens" in kw:
        kw = dict(kw, batch=len(kw["lens"]))
    wl = synth(**kw)
    run(wl, layout_every=2, cfg_overrides=_fp8_cfg(wl))


@needs_gpu
def test_fp8_kv_full_size_workload():
    wl = W.workload("llama3_8b_b1_128k")
    cfg = dict(kv_fp8=True, k_scale=[0.02 * (1 + h) for h in range(wl.Hkv)],
               v_scale=[0.05] * wl.Hkv)
    run(wl, steps=5, layout_every=4, cfg_overrides=cfg)


@needs_gpu
@pytest.mark.parametrize("which", ["synthetic", "many_clusters"])
def test_fp8_kv_statistics_and_page_mass(which):
    wl = PAGE_MASS_CASES[which]()
    pr = Pair(wl, cfg_overrides=_fp8_cfg(wl))
    for s in range(2):
        pr.step(s)
    q, _, _ = W.step_tokens(wl, 2)
    _check_page_mass(pr, q)
