"""Pins for the CPU oracle: every function checked against something other
than itself -- hand-worked fixtures (tests/golden/), closed forms, textbook
routines (torch SDPA in fp64 on the CPU, numpy reductions), invariants and
brute force on tiny inputs.  CPU only."""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for ln in f:
            ln = ln.strip()
            if ln and not ln.startswith("#"):
                yield ln


def f16(x):
    return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


# ---- exact decoding of the storage formats --------------------------------

def test_decode_all_f16_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.decode(bits, "f16")
    ok = np.isnan(ref) == np.isnan(got)
    assert ok.all()
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m])
    assert np.array_equal(np.signbit(got[m]), np.signbit(ref[m]))


def test_decode_all_bf16_patterns_match_float32_view():
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = oracle.decode(bits.astype(np.uint16), "bf16")
    m = ~np.isnan(ref)
    assert (np.isnan(got) == ~m).all()
    assert np.array_equal(got[m], ref[m])
    assert np.array_equal(np.signbit(got[m]), np.signbit(ref[m]))


def test_bf16_rounding_is_nearest_even():
    # generator rounding (not oracle arithmetic) must be RNE: torch's cast is
    # an independent implementation of the same rounding
    x = np.random.default_rng(1).standard_normal(100000).astype(np.float32)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 3.0e38]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(W.to_bits(x, "bf16"), ref.view(np.uint16))


# ---- metadata (min/max pooling per logical page) ---------------------------

def test_score_fixture_metadata_and_scores():
    d = ell = None
    q, k, kmin, kmax, s, S, maxdot = [], [], {}, {}, {}, {}, {}
    for ln in _lines("score_example.txt"):
        t = ln.split()
        if t[0] == "d":
            d = int(t[1])
        elif t[0] == "ell":
            ell = int(t[1])
        elif t[0] == "q":
            q.append([float(x) for x in t[1:]])
        elif t[0] == "k":
            k.append([float(x) for x in t[1:]])
        elif t[0] in ("kmin", "kmax"):
            (kmin if t[0] == "kmin" else kmax)[int(t[1])] = [float(x) for x in t[2:]]
        elif t[0] == "s":
            s[(int(t[1]), int(t[2]))] = float(t[3])
        elif t[0] == "S":
            S[int(t[1])] = float(t[2])
        elif t[0] == "maxdot":
            maxdot[(int(t[1]), int(t[2]))] = float(t[3])
    K = f16(k)
    mn, mx = oracle.page_minmax(K, "f16", ell)
    assert mn.shape == (2, d)
    for j in kmin:
        assert np.array_equal(oracle.decode(mn[j], "f16"), kmin[j])
        assert np.array_equal(oracle.decode(mx[j], "f16"), kmax[j])
    s64 = oracle.page_scores_f64(f16(q), mn, mx, "f16")
    for (h, j), v in s.items():
        assert s64[h, j] == v
    S32 = oracle.page_scores(f16(q), mn, mx, "f16")
    for j, v in S.items():
        assert S32[j] == np.float32(v)
    for (h, j), v in maxdot.items():
        assert v <= s64[h, j]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("L,ell", [(1, 16), (15, 16), (16, 16), (17, 16),
                                   (1000, 32), (4096, 64)])
def test_metadata_equals_numpy_reduction(dtype, L, ell):
    r = np.random.default_rng(L * 7 + ell)
    x = r.standard_normal((L, 24)).astype(np.float32)
    x[r.random(x.shape) < 0.05] = 0.0
    x[r.random(x.shape) < 0.05] *= -0.0
    K = W.to_bits(x, dtype)
    mn, mx = oracle.page_minmax(K, dtype, ell)
    vals = oracle.decode(K, dtype)
    nL = -(-L // ell)
    pad = nL * ell - L
    lo = np.concatenate([vals, np.full((pad, 24), np.inf)]).reshape(nL, ell, 24).min(1)
    hi = np.concatenate([vals, np.full((pad, 24), -np.inf)]).reshape(nL, ell, 24).max(1)
    assert np.array_equal(oracle.decode(mn, dtype), lo)
    assert np.array_equal(oracle.decode(mx, dtype), hi)


def test_metadata_incremental_equals_from_scratch():
    # the layer model recomputes only the pages touched by each append; that
    # must equal a from-scratch reduction over the whole key array
    cfg = dict(num_q_heads=4, num_kv_heads=2, head_dim=16, dtype="f16",
               logical_page=8, streaming=[False, False], max_context=200)
    lay = oracle.OracleLayer(cfg)
    sid = lay.new_seq()
    r = np.random.default_rng(5)
    for n in [1, 7, 8, 1, 30, 2, 64, 1, 1]:
        k = f16(r.standard_normal((n, 2, 16)))
        lay.append(sid, k, k)
    s = lay.seqs[sid]
    for h in (0, 1):
        mn, mx = oracle.page_minmax(s.K[h, :s.L], "f16", 8)
        assert np.array_equal(mn, s.kmin[h]) and np.array_equal(mx, s.kmax[h])


# ---- page score ------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_score_upper_bounds_every_token_dot(dtype):
    # closed-form invariant: q_c k_c <= max(q_c kmax_c, q_c kmin_c) for
    # k_c in [kmin_c, kmax_c], so s_h(j) >= max_{t in page j} q_h . k_t
    r = np.random.default_rng(11)
    L, d, ell, G = 1000, 64, 16, 4
    x = r.standard_normal((L, d)).astype(np.float32)
    x[:, [3, 40]] *= 50.0
    K = W.to_bits(x, dtype)
    q = W.to_bits(r.standard_normal((G, d)).astype(np.float32), dtype)
    mn, mx = oracle.page_minmax(K, dtype, ell)
    s = oracle.page_scores_f64(q, mn, mx, dtype)
    dots = oracle.decode(q, dtype) @ oracle.decode(K, dtype).T  # [G][L] fp64
    nL = mn.shape[0]
    for j in range(nL):
        best = dots[:, j * ell:min((j + 1) * ell, L)].max(axis=1)
        assert (s[:, j] >= best - 1e-9 * np.abs(best)).all()
    S = oracle.page_scores(q, mn, mx, dtype)
    assert np.allclose(S, s.max(0), rtol=1e-5, atol=1e-4)


def test_score_single_token_page_equals_dot():
    # a one-token page has kmin == kmax == k, so the score is exactly q . k
    r = np.random.default_rng(3)
    K = f16(r.standard_normal((5, 32)))
    q = f16(r.standard_normal((3, 32)))
    mn, mx = oracle.page_minmax(K, "f16", 1)
    s = oracle.page_scores_f64(q, mn, mx, "f16")
    ref = oracle.decode(q, "f16") @ oracle.decode(K, "f16").T
    assert np.allclose(s, ref, rtol=0, atol=1e-12)


def test_score_nonnegative_query_reads_kmax():
    r = np.random.default_rng(4)
    K = f16(r.standard_normal((64, 16)))
    q = f16(np.abs(r.standard_normal((2, 16))))
    mn, mx = oracle.page_minmax(K, "f16", 16)
    s = oracle.page_scores_f64(q, mn, mx, "f16")
    ref = oracle.decode(q, "f16") @ oracle.decode(mx, "f16").T
    assert np.allclose(s, ref, rtol=0, atol=1e-12)


def test_score_fp32_matches_numpy_fp64_expression():
    r = np.random.default_rng(6)
    K = f16(r.standard_normal((512, 128)))
    q = f16(r.standard_normal((4, 128)))
    mn, mx = oracle.page_minmax(K, "f16", 32)
    qv, lo, hi = (oracle.decode(a, "f16") for a in (q, mn, mx))
    ref = np.maximum(qv[:, None, :] * hi[None], qv[:, None, :] * lo[None]).sum(-1)
    S = oracle.page_scores(q, mn, mx, "f16")
    assert np.allclose(S, ref.max(0), rtol=1e-6, atol=1e-5)


def test_pins_catch_planted_score_mistakes():
    # plant plausible mistakes in the score (on the CPU) and check that a pin
    # rejects each: reading only kmin or a flipped sign breaks the upper
    # bound; a dropped channel breaks the single-token-page equality
    r = np.random.default_rng(12)
    K = f16(r.standard_normal((256, 32)))
    q = f16(r.standard_normal((2, 32)))
    mn, mx = oracle.page_minmax(K, "f16", 16)
    dots = oracle.decode(q, "f16") @ oracle.decode(K, "f16").T

    def bound_holds(s):
        return all((s[:, j] >= dots[:, j * 16:(j + 1) * 16].max(1) - 1e-9).all()
                   for j in range(16))

    assert bound_holds(oracle.page_scores_f64(q, mn, mx, "f16"))
    assert not bound_holds(oracle.page_scores_f64(q, mn, mn, "f16"))
    assert not bound_holds(-oracle.page_scores_f64(q, mx, mn, "f16"))
    m1, x1 = oracle.page_minmax(K, "f16", 1)
    exact = np.allclose(oracle.page_scores_f64(q, m1, x1, "f16"), dots, atol=1e-12)
    assert exact
    dropped = q.copy()
    dropped[:, -1] = 0
    assert not np.allclose(oracle.page_scores_f64(dropped, m1, x1, "f16"), dots,
                           atol=1e-12)


# ---- budget and top-k ------------------------------------------------------

def test_budget_fixture():
    for ln in _lines("budget_rule.txt"):
        L, tb, ell, pages = (int(x) for x in ln.split())
        assert oracle.budget_pages(L, tb, ell) == pages, ln


def test_selection_fixture():
    for ln in _lines("selection_example.txt"):
        a, b, c = ln.split("|")
        K_sel = int(a)
        S = np.array([float(x) for x in b.split()], np.float32)
        exp = [int(x) for x in c.split()]
        assert oracle.select(S, S.size, K_sel).tolist() == exp, ln


def _lexsort_select(S, nL, K_sel):
    if nL <= K_sel:
        return list(range(nL))
    j = np.arange(nL - 1)
    order = np.lexsort((j, -S[:nL - 1].astype(np.float64)))
    return sorted(order[:K_sel - 1].tolist() + [nL - 1])


@pytest.mark.parametrize("seed", range(8))
def test_selection_equals_lexsort(seed):
    r = np.random.default_rng(100 + seed)
    nL = int(r.integers(1, 3000))
    K_sel = int(r.integers(1, 200))
    S = r.integers(-20, 20, size=nL).astype(np.float32) * 0.25  # many ties
    if seed % 2:
        S = r.standard_normal(nL).astype(np.float32)
    got = oracle.select(S, nL, K_sel)
    assert got.tolist() == _lexsort_select(S, nL, K_sel)


@pytest.mark.parametrize("seed", range(30))
def test_selection_brute_force_tiny(seed):
    # enumerate every K_sel subset that contains the newest page; the chosen
    # one has the lexicographically best (descending score multiset, then
    # ascending indices) order
    r = np.random.default_rng(seed)
    nL = int(r.integers(2, 10))
    K_sel = int(r.integers(1, nL))
    S = r.integers(0, 4, size=nL).astype(np.float32)
    best = None
    for sub in itertools.combinations(range(nL - 1), K_sel - 1):
        key = (sorted((-S[j] for j in sub)), list(sub))
        if best is None or key < best[0]:
            best = (key, sorted(list(sub) + [nL - 1]))
    assert oracle.select(S, nL, K_sel).tolist() == best[1]


def test_newest_page_always_kept():
    S = np.array([5, 4, 3, 2, -100], np.float32)
    assert oracle.select(S, 5, 2).tolist() == [0, 4]


# ---- attended token sets ---------------------------------------------------

def test_token_set_fixture():
    for ln in _lines("token_sets.txt"):
        head, rest = ln.split("|", 1)
        h = head.split()
        if h[0] == "stream":
            L, S_, W_ = (int(x) for x in h[1:])
            exp = [int(x) for x in rest.split()]
            assert oracle.streaming_tokens(L, S_, W_).tolist() == exp, ln
        else:
            ell, L, nL0 = (int(x) for x in h[1:])
            sel_s, pos_s = rest.split("|")
            sel = [int(x) for x in sel_s.split()]
            exp = [int(x) for x in pos_s.split()]
            assert oracle.dynamic_tokens(sel, nL0, L, ell).tolist() == exp, ln


@pytest.mark.parametrize("L,S_,W_", [(5000, 128, 4096), (100, 16, 256),
                                     (4224, 128, 4096), (4225, 128, 4096)])
def test_streaming_set_closed_form(L, S_, W_):
    T = oracle.streaming_tokens(L, S_, W_)
    assert len(set(T.tolist())) == len(T)
    exp = min(L, S_ + W_)
    assert len(T) == exp


# ---- attention --------------------------------------------------------------

def _sdpa(q, K, V, dtype, mask=None):
    qv = torch.from_numpy(oracle.decode(q, dtype))[None, :, None, :]
    kv = torch.from_numpy(oracle.decode(K, dtype))[None, None]
    vv = torch.from_numpy(oracle.decode(V, dtype))[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None, None, :]
    G = q.shape[0]
    out = torch.nn.functional.scaled_dot_product_attention(
        qv, kv.expand(1, G, -1, -1), vv.expand(1, G, -1, -1), attn_mask=m)
    return out[0, :, 0].numpy()


def test_attention_fixture_closed_form():
    q = f16([[2, 0, 0, 0]])
    K = f16([[0, 0, 0, 0], [1, 0, 0, 0], [-1, 0, 0, 0]])
    V = f16([[1, 0, 0, 0], [0, 1, 0, 0], [0, 0, 1, 0]])
    # z = q.k / sqrt(4) = (0, 1, -1); weights proportional to (1, e, 1/e)
    den = 1 + math.e + 1 / math.e
    exp = np.array([1 / den, math.e / den, 1 / (math.e * den), 0.0])
    out = oracle.attention(q, K, V, "f16", [0, 1, 2])
    assert np.allclose(out[0], exp, rtol=0, atol=1e-15)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_dense_equivalence_with_sdpa(dtype):
    # budget >= L: every page is selected and the output is full attention
    r = np.random.default_rng(21)
    L, d, G = 700, 64, 4
    K = W.to_bits(r.standard_normal((L, d)).astype(np.float32), dtype)
    V = W.to_bits(r.standard_normal((L, d)).astype(np.float32), dtype)
    q = W.to_bits(r.standard_normal((G, d)).astype(np.float32), dtype)
    ell = 16
    nL = -(-L // ell)
    mn, mx = oracle.page_minmax(K, dtype, ell)
    sel = oracle.select(oracle.page_scores(q, mn, mx, dtype), nL,
                        oracle.budget_pages(L, L + 5, ell))
    assert sel.tolist() == list(range(nL))
    T = oracle.dynamic_tokens(sel, nL, L, ell)
    out = oracle.attention(q, K, V, dtype, T)
    assert np.allclose(out, _sdpa(q, K, V, dtype), rtol=0, atol=1e-12)


def test_streaming_equals_masked_sdpa():
    r = np.random.default_rng(22)
    L, d = 1500, 64
    K, V = (f16(r.standard_normal((L, d))) for _ in range(2))
    q = f16(r.standard_normal((2, d)))
    T = oracle.streaming_tokens(L, 16, 256)
    mask = np.zeros(L, bool)
    mask[:16] = True
    mask[L - 256:] = True
    out = oracle.attention(q, K, V, "f16", T)
    assert np.allclose(out, _sdpa(q, K, V, "f16", mask), rtol=0, atol=1e-12)


def test_sparse_equals_dense_with_mask():
    r = np.random.default_rng(23)
    L, d, ell = 2000, 32, 32
    K, V = (f16(r.standard_normal((L, d))) for _ in range(2))
    q = f16(r.standard_normal((4, d)))
    sel = np.sort(r.choice(-(-L // ell) - 1, size=9, replace=False)).astype(np.int32)
    sel = np.concatenate([sel, [-(-L // ell) - 1]]).astype(np.int32)
    T = oracle.dynamic_tokens(sel, -(-L // ell), L, ell)
    mask = np.zeros(L, bool)
    mask[T] = True
    assert mask.sum() == len(T)
    out = oracle.attention(q, K, V, "f16", T)
    assert np.allclose(out, _sdpa(q, K, V, "f16", mask), rtol=0, atol=1e-12)


def test_special_cases():
    r = np.random.default_rng(24)
    d = 64
    V = f16(r.standard_normal((50, d)))
    K = f16(r.standard_normal((50, d)))
    q = f16(r.standard_normal((2, d)))
    # one token: out = v_0
    out = oracle.attention(q, K, V, "f16", [0])
    assert np.array_equal(out, np.repeat(oracle.decode(V[:1], "f16"), 2, 0))
    # identical keys: uniform weights, out = mean of V over the set
    Ks = np.repeat(K[:1], 50, 0)
    T = np.arange(3, 40)
    out = oracle.attention(q, Ks, V, "f16", T)
    assert np.allclose(out, oracle.decode(V[T], "f16").mean(0)[None], atol=1e-12)
    # a needle with a huge logit takes all the weight
    Kn = K.copy()
    qd = oracle.decode(q[:1], "f16")[0]
    Kn[17] = f16(60.0 * qd / np.linalg.norm(qd))
    out = oracle.attention(q[:1], Kn, V, "f16", np.arange(50))
    assert np.allclose(out[0], oracle.decode(V[17], "f16"), atol=1e-6)


# ---- selection reuse over decode steps --------------------------------------

def _tiny_layer(C=4, budget=64, streaming=(False, True)):
    cfg = dict(num_q_heads=4, num_kv_heads=2, head_dim=16, dtype="f16",
               logical_page=8, streaming=list(streaming), sink=4, window=24,
               token_budget=budget, reuse_interval=C, max_context=2000)
    return oracle.OracleLayer(cfg)


def test_selection_reused_for_C_steps_and_tail_pages_attended():
    lay = _tiny_layer()
    sid = lay.new_seq()
    r = np.random.default_rng(30)
    ctx = f16(r.standard_normal((301, 2, 16)))
    lay.append(sid, ctx, ctx)
    ran, sels = [], []
    for step in range(13):
        q = f16(r.standard_normal((4, 16)))
        kv = f16(r.standard_normal((2, 16)))
        lay.append(sid, kv[None], kv[None])
        ran.append(lay.select(sid, q))
        sels.append(lay.seqs[sid].sel[0].copy())
        nL = -(-lay.seqs[sid].L // 8)
        T = set(lay.tokens(sid, 0).tolist())
        # every page from the selection-time last page to the current last
        # page is attended, whatever the stored selection holds
        for j in range(lay.seqs[sid].nL0[0] - 1, nL):
            assert set(range(j * 8, min((j + 1) * 8, lay.seqs[sid].L))) <= T
        lay.attend(sid, q)
    assert ran == [s % 4 == 0 for s in range(13)]
    for s in range(13):
        if s % 4:
            assert np.array_equal(sels[s], sels[s - s % 4])
    # a page boundary was crossed inside a reuse window (L 302..314, ell 8)
    assert any(not ran[s] and (302 + s) % 8 == 1 for s in range(13))


def test_layer_step_dense_when_budget_covers_context():
    lay = _tiny_layer(budget=10 ** 6, streaming=(False, False))
    sid = lay.new_seq()
    r = np.random.default_rng(31)
    ctx = f16(r.standard_normal((120, 2, 16)))
    vv = f16(r.standard_normal((120, 2, 16)))
    lay.append(sid, ctx, vv)
    q = f16(r.standard_normal((4, 16)))
    lay.select(sid, q)
    out = lay.attend(sid, q)
    for h in range(2):
        ref = _sdpa(q[2 * h:2 * h + 2], ctx[:, h], vv[:, h], "f16")
        assert np.allclose(out[2 * h:2 * h + 2], ref, atol=1e-12)


# ---- softmax statistics (row max, row sum) --------------------------------

def test_softmax_stats_closed_forms():
    # z = q.k / sqrt(4) = (0, 1, -1): max 1, sum 1/e + 1 + 1/e^2
    q = f16([[2, 0, 0, 0]])
    K = f16([[0, 0, 0, 0], [1, 0, 0, 0], [-1, 0, 0, 0]])
    rm, rs = oracle.softmax_stats(q, K, "f16", [0, 1, 2])
    assert rm[0] == 1.0
    assert rs[0] == pytest.approx(math.exp(-1) + 1 + math.exp(-2), rel=1e-15)
    # one token: the sum is exactly 1 and the max is that token's logit
    rm, rs = oracle.softmax_stats(q, K, "f16", [2])
    assert (rm[0], rs[0]) == (-1.0, 1.0)
    # n identical keys: every logit equals the max, the sum is n
    Kc = f16([[0.5, -1, 2, 0]] * 9)
    rm, rs = oracle.softmax_stats(q, Kc, "f16", list(range(9)))
    assert (rm[0], rs[0]) == (0.5, 9.0)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_softmax_stats_match_a_library_logsumexp(dtype):
    # log(row_sum) + row_max is the log-sum-exp of the logits: compare with
    # torch.logsumexp over logits computed independently (fp64 matmul)
    r = np.random.default_rng(23)
    L, d, G = 500, 64, 4
    K = W.to_bits(r.standard_normal((L, d)).astype(np.float32), dtype)
    q = W.to_bits(r.standard_normal((G, d)).astype(np.float32), dtype)
    T = np.sort(r.choice(L, 123, replace=False)).astype(np.int32)
    rm, rs = oracle.softmax_stats(q, K, dtype, T)
    z = (torch.from_numpy(oracle.decode(q, dtype)) @
         torch.from_numpy(oracle.decode(K, dtype))[T].T) / math.sqrt(d)
    assert np.allclose(rm, z.max(dim=1).values.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(np.log(rs) + rm, torch.logsumexp(z, dim=1).numpy(), rtol=0, atol=1e-12)


def test_page_mass_closed_forms():
    # z = q.k / sqrt(4) over tokens 0..5 with ell = 2 (pages 0, 1, 2):
    # logits (0, 1, -1, 0, 1, 1); every page's mass is its share of exp(z)
    q = f16([[2, 0, 0, 0]])
    K = f16([[0, 0, 0, 0], [1, 0, 0, 0], [-1, 0, 0, 0], [0, 0, 0, 0], [1, 0, 0, 0],
             [1, 0, 0, 0]])
    e = [math.exp(z) for z in (0, 1, -1, 0, 1, 1)]
    den = sum(e)
    m = oracle.page_mass(q, K, "f16", list(range(6)), 2, [0, 1, 2])
    assert m[0] == pytest.approx([(e[0] + e[1]) / den, (e[2] + e[3]) / den,
                                  (e[4] + e[5]) / den], rel=1e-14)
    # a page outside the attended tokens has no mass; a page missing from the
    # list takes its tokens' weight with it
    m = oracle.page_mass(q, K, "f16", [0, 1, 4, 5], 2, [0, 1, 2])
    assert m[0][1] == 0.0 and m[0][0] + m[0][2] == pytest.approx(1.0, abs=1e-15)
    m = oracle.page_mass(q, K, "f16", list(range(6)), 2, [2])
    assert m[0][0] == pytest.approx((e[4] + e[5]) / den, rel=1e-14)
    # one token: all the mass on its page
    assert oracle.page_mass(q, K, "f16", [3], 2, [1]).tolist() == [[1.0]]


def test_page_mass_equal_keys_count_tokens():
    # identical keys: every attended token has weight 1/|T|, so a page's mass
    # is its attended token count over |T| (a partial last page included)
    ell, L = 16, 100
    K = f16([[0.25, -1, 2, 0.5]] * L)
    q = f16([[1, 2, -0.5, 3], [-2, 0, 1, 1]])
    T = np.concatenate([np.arange(0, 20), np.arange(40, 48), np.arange(90, 100)])
    pages = [0, 1, 2, 5, 6]
    m = oracle.page_mass(q, K, "f16", T, ell, pages)
    want = np.array([np.sum(T // ell == j) for j in pages]) / T.size
    assert np.allclose(m, want[None, :], rtol=0, atol=1e-15)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_page_mass_matches_a_library_softmax(dtype):
    # every page attended: the masses are torch.softmax over all L logits
    # (fp64 matmul), summed over each page's ell columns
    r = np.random.default_rng(29)
    L, d, G, ell = 300, 64, 4, 16
    K = W.to_bits(r.standard_normal((L, d)).astype(np.float32), dtype)
    q = W.to_bits(r.standard_normal((G, d)).astype(np.float32), dtype)
    nL = -(-L // ell)
    m = oracle.page_mass(q, K, dtype, np.arange(L), ell, np.arange(nL))
    z = (torch.from_numpy(oracle.decode(q, dtype)) @
         torch.from_numpy(oracle.decode(K, dtype)).T) / math.sqrt(d)
    w = torch.nn.functional.pad(torch.softmax(z, dim=1), (0, nL * ell - L))
    assert np.allclose(m, w.reshape(G, nL, ell).sum(-1).numpy(), rtol=0, atol=1e-14)
    assert np.allclose(m.sum(1), 1.0, rtol=0, atol=1e-13)


def test_page_mass_of_a_decode_layer():
    # the decode state's attended pages are the selection plus the pages
    # created since; a planted needle page takes nearly all the mass
    cfg = dict(num_q_heads=2, num_kv_heads=1, head_dim=64, dtype="bf16", logical_page=16,
               streaming=[False], sink=0, window=0, token_budget=64, reuse_interval=4,
               max_context=4096)
    r = np.random.default_rng(31)
    orc = oracle.OracleLayer(cfg)
    sid = orc.new_seq()
    L = 1000
    Kf = r.standard_normal((L, 1, 64)).astype(np.float32) * 0.1
    u = r.standard_normal(64).astype(np.float32)
    Kf[320:336, 0] = 8 * u / np.linalg.norm(u)          # page 20
    K = W.to_bits(Kf, "bf16")
    V = W.to_bits(r.standard_normal((L, 1, 64)).astype(np.float32), "bf16")
    orc.append(sid, K, V)
    q = W.to_bits(np.stack([u, u]), "bf16")
    orc.select(sid, q)
    orc.append(sid, K[:20], V[:20])                      # 20 more tokens: a new page
    pages, mass = orc.page_mass(sid, q)[0]
    sel = orc.seqs[sid].sel[0]
    assert 20 in sel and sel[-1] == 62
    assert pages.tolist() == sorted(set(sel.tolist()) | {62, 63})
    assert mass.shape == (2, pages.size)
    assert np.allclose(mass.sum(1), 1.0, atol=1e-13)
    assert np.all(mass[:, pages.tolist().index(20)] > 0.9)


# ---- fp8 (e4m3) KV storage ------------------------------------------------------

def _torch_e4m3(codes):
    """Library decode of e4m3 codes (torch's float8_e4m3fn)."""
    c = torch.from_numpy(np.asarray(codes, np.uint8).copy())
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_all_codes_match_the_library():
    codes = np.arange(256)
    got = oracle.e4m3_value(codes)
    ref = _torch_e4m3(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m])
    # the format's landmarks
    assert oracle.e4m3_value([0x7E, 0x08, 0x01, 0x38, 0xB8]).tolist() == \
        [448.0, 2.0 ** -6, 2.0 ** -9, 1.0, -1.0]
    assert np.isnan(oracle.e4m3_value([0x7F, 0xFF])).all()


def test_e4m3_encode_rounds_like_the_library_and_saturates():
    r = np.random.default_rng(41)
    grid = _torch_e4m3(np.arange(0x7F))                   # every finite magnitude
    mids = (grid[:-1] + grid[1:]) / 2                     # exact ties
    x = np.concatenate([grid, mids, -mids, r.uniform(-448, 448, 4000),
                        r.standard_normal(2000) * 1e-2, np.float32(2.0 ** -10) * np.arange(9)])
    x = x.astype(np.float32)
    got = oracle.e4m3_from_float(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    # saturation (finite clamp) above the largest magnitude, and NaN
    big = np.array([448.0, 449.0, 463.9, 464.0, 1e4, np.inf], np.float32)
    assert oracle.e4m3_from_float(big).tolist() == [0x7E] * 6
    assert oracle.e4m3_from_float(-big).tolist() == [0xFE] * 6
    assert oracle.e4m3_from_float([np.nan]).tolist() == [0x7F]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_e4m3_quantize_divides_once_in_fp32(dtype):
    r = np.random.default_rng(43)
    xb = W.to_bits((r.standard_normal(5000) * 3).astype(np.float32), dtype)
    scale = np.float32(0.0371)
    got = oracle.quantize_e4m3(xb, dtype, scale)
    t = torch.from_numpy(oracle.decode(xb, dtype).astype(np.float32)) / float(scale)
    ref = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    # a value that is exactly scale * code comes back as that code
    assert oracle.quantize_e4m3(W.to_bits(np.float32([0.5]), dtype), dtype, 0.25).tolist() == \
        [0x40]


def test_fp8_scores_scale_with_the_key_scale_and_bound_the_keys():
    r = np.random.default_rng(45)
    L, d, G, ell = 160, 64, 2, 16
    K = r.integers(0, 0x7F, (L, d)) | (r.integers(0, 2, (L, d)) << 7)
    K = K.astype(np.uint16)
    q = W.to_bits(r.standard_normal((G, d)).astype(np.float32), "bf16")
    mn, mx = oracle.page_minmax(K, "e4m3", ell)
    s1 = oracle.page_scores(q, mn, mx, "bf16", "e4m3", 1.0)
    s2 = oracle.page_scores(q, mn, mx, "bf16", "e4m3", 2.0)
    assert np.array_equal(s2, 2 * s1)
    # upper bound: s_h(j) >= q_h . k_t for every token of page j (fp64)
    ks = 0.75
    s64 = oracle.page_scores_f64(q, mn, mx, "bf16", "e4m3", ks)
    dots = oracle.decode(q, "bf16") @ (ks * oracle.e4m3_value(K)).T   # [G][L]
    for j in range(L // ell):
        assert np.all(s64[:, j] >= dots[:, j * ell:(j + 1) * ell].max(1) - 1e-12)


def test_fp8_decode_layer_is_sdpa_over_dequantized_kv():
    # budget >= L, no streaming head: the fp8 layer attends every token of
    # the quantised cache -- torch SDPA over the dequantised values, where the
    # codes come from the library's own fp32 division and e4m3 rounding
    r = np.random.default_rng(47)
    L, d, Hkv, G = 300, 64, 2, 2
    ks, vs = [0.02, 0.5], [0.125, 3.0]
    cfg = dict(num_q_heads=Hkv * G, num_kv_heads=Hkv, head_dim=d, dtype="bf16",
               logical_page=16, streaming=[False] * Hkv, sink=0, window=0,
               token_budget=10 ** 6, reuse_interval=4, max_context=1024,
               kv_fp8=True, k_scale=ks, v_scale=vs)
    orc = oracle.OracleLayer(cfg)
    sid = orc.new_seq()
    K = W.to_bits(r.standard_normal((L, Hkv, d)).astype(np.float32), "bf16")
    V = W.to_bits(r.standard_normal((L, Hkv, d)).astype(np.float32), "bf16")
    q = W.to_bits(r.standard_normal((Hkv * G, d)).astype(np.float32), "bf16")
    orc.append(sid, K, V)
    orc.select(sid, q)
    out = orc.attend(sid, q)

    def deq(bits, scale):
        t = torch.from_numpy(oracle.decode(bits, "bf16").astype(np.float32)) / np.float32(scale)
        return t.to(torch.float8_e4m3fn).to(torch.float64) * float(np.float32(scale))

    qd = torch.from_numpy(oracle.decode(q, "bf16"))
    for h in range(Hkv):
        kd, vd = deq(K[:, h], ks[h]), deq(V[:, h], vs[h])
        ref = torch.nn.functional.scaled_dot_product_attention(
            qd[h * G:(h + 1) * G][None, :, None, :], kd[None, None].expand(1, G, -1, -1),
            vd[None, None].expand(1, G, -1, -1))[0, :, 0].numpy()
        assert np.allclose(out[h * G:(h + 1) * G], ref, rtol=0, atol=1e-12), h
    # the stored codes and the page metadata are the quantised keys
    s = orc.seqs[sid]
    assert np.array_equal(s.K[0, :L], oracle.quantize_e4m3(K[:, 0], "bf16", ks[0]))
    mn, mx = oracle.page_minmax(s.K[1, :L], "e4m3", 16)
    assert np.array_equal(s.kmin[1], mn) and np.array_equal(s.kmax[1], mx)


# ---- prefill: low-rank block importance, block-sparse causal attention ----------

def _prefill_inputs(seed, L, d, G, r, dtype="bf16"):
    rg = np.random.default_rng(seed)
    Q = W.to_bits(rg.standard_normal((G, L, d)).astype(np.float32), dtype)
    K = W.to_bits(rg.standard_normal((L, d)).astype(np.float32), dtype)
    V = W.to_bits(rg.standard_normal((L, d)).astype(np.float32), dtype)
    Wq = (rg.standard_normal((d, r)) / math.sqrt(d)).astype(np.float32)
    Wk = (rg.standard_normal((d, r)) / math.sqrt(d)).astype(np.float32)
    return Q, K, V, Wq, Wk


def test_prefill_block_scores_equal_the_pairwise_mean():
    # the definition: mean over the block pair's token pairs of the low-rank
    # logits, max over the group -- brute force with torch, partial last block
    L, d, G, r, blk = 150, 64, 2, 8, 32
    Q, K, _, Wq, Wk = _prefill_inputs(51, L, d, G, r)
    S = oracle.prefill_block_scores(Q, K, "bf16", Wq, Wk, blk)
    qt = torch.from_numpy(oracle.decode(Q, "bf16")) @ torch.from_numpy(Wq).double()
    kt = torch.from_numpy(oracle.decode(K, "bf16")) @ torch.from_numpy(Wk).double()
    z = qt @ kt.T / math.sqrt(d)                                  # [G][L][L]
    nb = -(-L // blk)
    for b in range(nb):
        for i in range(nb):
            if i > b:
                assert S[b, i] == -np.inf
                continue
            m = z[:, b * blk:(b + 1) * blk, i * blk:(i + 1) * blk].mean(dim=(1, 2))
            assert abs(S[b, i] - float(m.max())) <= 1e-12, (b, i)


def test_prefill_identity_projection_scores_mean_exact_logits():
    L, d, G, blk = 96, 16, 1, 32
    Q, K, _, _, _ = _prefill_inputs(53, L, d, G, 2, "f16")
    eye = np.eye(d, dtype=np.float32)
    S = oracle.prefill_block_scores(Q, K, "f16", eye, eye, blk)
    z = (torch.from_numpy(oracle.decode(Q, "f16"))[0] @
         torch.from_numpy(oracle.decode(K, "f16")).T) / math.sqrt(d)
    assert abs(S[2, 1] - float(z[64:96, 32:64].mean())) <= 1e-12


def _block_mask(blocks, blk, L):
    M = np.zeros((L, L), bool)
    for b, sel in enumerate(blocks):
        for t in range(b * blk, min((b + 1) * blk, L)):
            for i in sel:
                s0, s1 = i * blk, min((i + 1) * blk, t + 1)
                if s1 > s0:
                    M[t, s0:s1] = True
    return M


def _sdpa_masked(Q, K, V, dtype, M):
    q = torch.from_numpy(oracle.decode(Q, dtype))[None]            # [1][G][L][d]
    k = torch.from_numpy(oracle.decode(K, dtype))[None, None].expand(1, Q.shape[0], -1, -1)
    v = torch.from_numpy(oracle.decode(V, dtype))[None, None].expand(1, Q.shape[0], -1, -1)
    return torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=torch.from_numpy(M)[None, None])[0].numpy()


def test_prefill_below_the_dense_threshold_is_causal_attention():
    L, d, G, r, blk = 200, 32, 2, 4, 32
    Q, K, V, Wq, Wk = _prefill_inputs(55, L, d, G, r)
    S = oracle.prefill_block_scores(Q, K, "bf16", Wq, Wk, blk)
    blocks = oracle.prefill_select(S, blk, L, token_budget=32, dense_below=32768)
    assert [b.tolist() for b in blocks] == [list(range(b + 1)) for b in range(len(blocks))]
    out = oracle.prefill_attention(Q, K, V, "bf16", blocks, blk)
    q = torch.from_numpy(oracle.decode(Q, "bf16"))[None]
    k = torch.from_numpy(oracle.decode(K, "bf16"))[None, None].expand(1, G, -1, -1)
    v = torch.from_numpy(oracle.decode(V, "bf16"))[None, None].expand(1, G, -1, -1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)[0].numpy()
    assert np.allclose(out, ref, rtol=0, atol=1e-12)


def test_prefill_sparse_blocks_are_block_masked_attention():
    L, d, G, r, blk = 480, 32, 2, 4, 32
    Q, K, V, Wq, Wk = _prefill_inputs(57, L, d, G, r)
    S = oracle.prefill_block_scores(Q, K, "bf16", Wq, Wk, blk)
    blocks = oracle.prefill_select(S, blk, L, token_budget=4 * blk, dense_below=256)
    for b, sel in enumerate(blocks):
        assert b in sel and np.all(np.diff(sel) > 0) and len(sel) == min(b + 1, 4)
        if b >= 4:   # the best three earlier blocks by (score desc, index asc)
            order = np.lexsort((np.arange(b), -S[b, :b].astype(np.float32)))
            assert sorted(order[:3].tolist()) == [i for i in sel.tolist() if i != b]
    out = oracle.prefill_attention(Q, K, V, "bf16", blocks, blk)
    ref = _sdpa_masked(Q, K, V, "bf16", _block_mask(blocks, blk, L))
    assert np.allclose(out, ref, rtol=0, atol=1e-12)


def test_prefill_planted_block_is_chosen():
    # a key block aligned with every query's projected direction outranks
    # the rest for all later query blocks
    L, d, G, r, blk = 640, 32, 1, 4, 32
    _, K, _, Wq, Wk = _prefill_inputs(59, L, d, G, r)
    rg = np.random.default_rng(60)
    c = rg.standard_normal(d).astype(np.float32)                 # queries share a direction
    Q = W.to_bits((c + 0.5 * rg.standard_normal((G, L, d))).astype(np.float32), "bf16")
    Kf = oracle.decode(K, "bf16").astype(np.float32)
    u = c @ Wq @ Wk.T                                            # the key the scores reward
    Kf[96:128] = 6 * u / np.linalg.norm(u)
    K2 = W.to_bits(Kf, "bf16")
    S = oracle.prefill_block_scores(Q, K2, "bf16", Wq, Wk, blk)
    blocks = oracle.prefill_select(S, blk, L, token_budget=2 * blk, dense_below=0)
    assert all(3 in sel for sel in blocks[4:])


def test_prefill_attention_is_the_per_token_attention():
    # the prompt routine equals `attention` called once per query token on
    # its allowed keys, bit for bit (same products in the same order)
    L, d, G, blk = 200, 32, 2, 32
    Q, K, V, Wq, Wk = _prefill_inputs(61, L, d, G, 4, "f16")
    S = oracle.prefill_block_scores(Q, K, "f16", Wq, Wk, blk)
    blocks = oracle.prefill_select(S, blk, L, token_budget=2 * blk, dense_below=0)
    out = oracle.prefill_attention(Q, K, V, "f16", blocks, blk)
    for t in (0, 31, 32, 100, 199):
        sel = blocks[t // blk]
        toks = np.concatenate([np.arange(i * blk, min((i + 1) * blk, L)) for i in sel])
        ref = oracle.attention(Q[:, t], K, V, "f16", toks[toks <= t])
        assert np.array_equal(out[:, t], ref), t
