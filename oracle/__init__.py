"""Plain CPU oracle for LServe-style decode-phase sparse attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check in
``__graft_entry__`` and by the CPU-baseline leg of ``bench.py``.  The product
path (the CUDA library and its binding) never imports it.

Two layers:

* ``liboracle.so`` (``spd_oracle.c``): the arithmetic, written out from the
  definitions (page min/max, page score, top-k under a budget, attended
  token sets, two-pass fp64 softmax attention, the softmax row max / row
  sum and the per-page attention mass).  Thin ctypes wrappers below.
* ``OracleLayer``: the per-sequence decode state on logical positions --
  length, the step counter that drives selection reuse every C steps, the
  page count at the last selection and the stored selection.  Plain Python
  control flow around the C arithmetic.

Sources ("LServe long-sequence LLM serving system" write-up unless noted):
  section 2.1  streaming heads, dynamic query-aware selection with a token
               budget (default 4096), min-max pooling of key blocks;
  section 2.2  hierarchical paging: logical pages of 16-64 tokens;
  section 3.2  reusable page selector (C = 4), dynamic budget
               min(4096, length/32);
  "Long-context inference optimization for LLMs" survey, section 2.2
               (StreamingLLM = attention sink + local window; Quest =
               query-aware block importance) and section 2.3 (GQA head
               sharing, 1/sqrt(head_dim) scale).

Readings where the pages are silent:
  the group score is the max over the G query heads sharing a kv head; the
  page holding the newest token is always kept; pages created during a
  reuse window are attended; the window includes the newest token and sink
  and window never double-count a position; the output is fp32/fp64.

Pins: tests/test_oracle_pins.py checks every function here against closed
forms, textbook routines (torch SDPA in fp64), brute force and hand-worked
fixtures in tests/golden/.
"""
import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

F16, BF16, E4M3 = 0, 1, 2
_DTYPES = {"f16": F16, "fp16": F16, "float16": F16,
           "bf16": BF16, "bfloat16": BF16, "e4m3": E4M3}

_lib = None


def lib():
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
        f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
        i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
        ci, cl = ctypes.c_int, ctypes.c_long
        L.orc_value.argtypes = [ctypes.c_uint16, ci]
        L.orc_value.restype = ctypes.c_double
        L.orc_decode.argtypes = [u16p, ci, cl, f64p]
        L.orc_decode.restype = None
        L.orc_page_minmax.argtypes = [u16p, ci, ci, ci, ci, ci, ci, u16p, u16p]
        L.orc_page_minmax.restype = ci
        L.orc_page_scores_f32.argtypes = [u16p, u16p, u16p, ci, ci, ci, ci, f32p]
        L.orc_page_scores_f32.restype = None
        L.orc_page_scores_f64.argtypes = [u16p, u16p, u16p, ci, ci, ci, ci, f64p]
        L.orc_page_scores_f64.restype = None
        L.orc_budget_pages.argtypes = [cl, ci, ci]
        L.orc_budget_pages.restype = ci
        L.orc_select.argtypes = [f32p, ci, ci, i32p]
        L.orc_select.restype = ci
        L.orc_dynamic_tokens.argtypes = [i32p, ci, ci, cl, ci, i32p]
        L.orc_dynamic_tokens.restype = ci
        L.orc_streaming_tokens.argtypes = [cl, ci, ci, i32p]
        L.orc_streaming_tokens.restype = ci
        L.orc_attention.argtypes = [u16p, u16p, u16p, ci, ci, ci, i32p, ci, f64p]
        L.orc_attention.restype = ci
        L.orc_softmax_stats.argtypes = [u16p, u16p, ci, ci, ci, i32p, ci, f64p, f64p]
        L.orc_softmax_stats.restype = ci
        L.orc_page_mass.argtypes = [u16p, u16p, ci, ci, ci, i32p, ci, ci, i32p, ci, f64p]
        L.orc_page_mass.restype = ci
        f32, f64 = ctypes.c_float, ctypes.c_double
        L.orc_e4m3_value.argtypes = [ctypes.c_uint]
        L.orc_e4m3_value.restype = f64
        L.orc_e4m3_from_float.argtypes = [f32]
        L.orc_e4m3_from_float.restype = ctypes.c_uint
        L.orc_quantize_e4m3.argtypes = [u16p, ci, cl, f32, u16p]
        L.orc_quantize_e4m3.restype = None
        L.orc_page_scores_f32_kv.argtypes = [u16p, ci, u16p, u16p, ci, f64, ci, ci, ci, f32p]
        L.orc_page_scores_f32_kv.restype = None
        L.orc_page_scores_f64_kv.argtypes = [u16p, ci, u16p, u16p, ci, f64, ci, ci, ci, f64p]
        L.orc_page_scores_f64_kv.restype = None
        L.orc_attention_kv.argtypes = [u16p, ci, u16p, u16p, ci, f64, f64, ci, ci, i32p, ci,
                                       f64p]
        L.orc_attention_kv.restype = ci
        L.orc_softmax_stats_kv.argtypes = [u16p, ci, u16p, ci, f64, ci, ci, i32p, ci, f64p,
                                           f64p]
        L.orc_softmax_stats_kv.restype = ci
        L.orc_page_mass_kv.argtypes = [u16p, ci, u16p, ci, f64, ci, ci, i32p, ci, ci, i32p, ci,
                                       f64p]
        L.orc_page_mass_kv.restype = ci
        L.orc_prefill_block_scores.argtypes = [u16p, ci, u16p, ci, f64, f32p, f32p, ci, ci, ci,
                                               ci, ci, f64p]
        L.orc_prefill_block_scores.restype = ci
        L.orc_prefill_attention.argtypes = [u16p, ci, u16p, u16p, ci, f64, f64, ci, ci, ci, ci,
                                            i32p, i32p, f64p]
        L.orc_prefill_attention.restype = ci
        _lib = L
    return _lib


def dtype_code(dtype):
    return _DTYPES[dtype] if isinstance(dtype, str) else int(dtype)


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


# ---- thin wrappers over the C arithmetic -----------------------------------

def decode(bits, dtype):
    """Exact value (fp64) of fp16/bf16 bit patterns."""
    b = _u16(bits)
    out = np.empty(b.shape, np.float64)
    lib().orc_decode(b.reshape(-1), dtype_code(dtype), b.size, out.reshape(-1))
    return out


def page_minmax(K, dtype, ell, j0=0, j1=None):
    """Per logical page min/max bit patterns of K [L][d] for pages [j0, j1)."""
    K = _u16(K)
    L, d = K.shape
    nL = -(-L // ell)
    j1 = nL if j1 is None else j1
    kmin = np.empty((j1 - j0, d), np.uint16)
    kmax = np.empty((j1 - j0, d), np.uint16)
    rc = lib().orc_page_minmax(K, dtype_code(dtype), L, d, ell, j0, j1, kmin, kmax)
    if rc != 0:
        raise ValueError("orc_page_minmax: bad arguments")
    return kmin, kmax


def e4m3_value(codes):
    """Exact value (fp64) of fp8 e4m3 codes."""
    c = np.asarray(codes).reshape(-1)
    return np.array([lib().orc_e4m3_value(int(x) & 0xff) for x in c],
                    np.float64).reshape(np.shape(codes))


def e4m3_from_float(x):
    """Codes of fp32 values, rounded to nearest even, saturating at +-448."""
    x = np.asarray(x, np.float32)
    return np.array([lib().orc_e4m3_from_float(float(v)) for v in x.reshape(-1)],
                    np.uint16).reshape(x.shape)


def quantize_e4m3(x, dtype, scale):
    """fp8 KV codes of 16-bit values x: e4m3(fl32(x / scale)), in uint16."""
    x = _u16(x)
    out = np.empty(x.shape, np.uint16)
    lib().orc_quantize_e4m3(x.reshape(-1), dtype_code(dtype), x.size, float(scale),
                            out.reshape(-1))
    return out


def _kv(dtype, kv_dtype):
    return dtype_code(dtype), dtype_code(dtype if kv_dtype is None else kv_dtype)


def page_scores(q, kmin, kmax, dtype, kv_dtype=None, kscale=1.0):
    """fp32 kv-head score S[nL] = max over the G query heads of q [G][d];
    kmin/kmax are kv_dtype codes of value / kscale (default: q's dtype, 1)."""
    q, kmin, kmax = _u16(q), _u16(kmin), _u16(kmax)
    G, d = q.shape
    nL = kmin.shape[0]
    S = np.empty(nL, np.float32)
    qd, kd = _kv(dtype, kv_dtype)
    lib().orc_page_scores_f32_kv(q, qd, kmin, kmax, kd, float(kscale), nL, G, d, S)
    return S


def page_scores_f64(q, kmin, kmax, dtype, kv_dtype=None, kscale=1.0):
    """fp64 per-head score s[G][nL] (not reduced over the group)."""
    q, kmin, kmax = _u16(q), _u16(kmin), _u16(kmax)
    G, d = q.shape
    nL = kmin.shape[0]
    s = np.empty((G, nL), np.float64)
    qd, kd = _kv(dtype, kv_dtype)
    lib().orc_page_scores_f64_kv(q, qd, kmin, kmax, kd, float(kscale), nL, G, d, s)
    return s


def budget_pages(L, token_budget, ell):
    return int(lib().orc_budget_pages(int(L), int(token_budget), int(ell)))


def select(S, nL, K_sel):
    """Sorted selection of logical pages (see orc_select)."""
    S = np.ascontiguousarray(S, dtype=np.float32)
    if S.shape[0] < nL:
        S = np.concatenate([S, np.zeros(nL - S.shape[0], np.float32)])
    sel = np.empty(max(K_sel, 1), np.int32)
    n = lib().orc_select(S, int(nL), int(K_sel), sel)
    if n < 0:
        raise ValueError("orc_select: bad arguments")
    return sel[:n].copy()


def dynamic_tokens(sel, nL0, L, ell):
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    out = np.empty(max(int(L), 1), np.int32)
    n = lib().orc_dynamic_tokens(sel, sel.size, int(nL0), int(L), int(ell), out)
    if n < 0:
        raise ValueError("orc_dynamic_tokens: bad arguments")
    return out[:n].copy()


def streaming_tokens(L, sink, window):
    out = np.empty(max(int(L), 1), np.int32)
    n = lib().orc_streaming_tokens(int(L), int(sink), int(window), out)
    return out[:n].copy()


def attention(q, K, V, dtype, tokens, kv_dtype=None, kscale=1.0, vscale=1.0):
    """fp64 softmax attention of q [G][d] over rows `tokens` of K/V [L][d]
    (kv_dtype codes of value / kscale, value / vscale; default q's dtype, 1)."""
    q, K, V = _u16(q), _u16(K), _u16(V)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    G, d = q.shape
    out = np.empty((G, d), np.float64)
    qd, kd = _kv(dtype, kv_dtype)
    if lib().orc_attention_kv(q, qd, K, V, kd, float(kscale), float(vscale), G, d, tokens,
                              tokens.size, out) != 0:
        raise ValueError("orc_attention: empty token set")
    return out


def softmax_stats(q, K, dtype, tokens, kv_dtype=None, kscale=1.0):
    """fp64 (row_max [G], row_sum [G]) of the logits q . k_t / sqrt(d) over
    rows `tokens` of K [L][d]: the max and the sum of exp(z - max)."""
    q, K = _u16(q), _u16(K)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    G, d = q.shape
    rm = np.empty(G, np.float64)
    rs = np.empty(G, np.float64)
    qd, kd = _kv(dtype, kv_dtype)
    if lib().orc_softmax_stats_kv(q, qd, K, kd, float(kscale), G, d, tokens, tokens.size, rm,
                                  rs) != 0:
        raise ValueError("orc_softmax_stats: empty token set")
    return rm, rs


def page_mass(q, K, dtype, tokens, ell, pages, kv_dtype=None, kscale=1.0):
    """fp64 [G][len(pages)]: the softmax weight of the logits q . k_t / sqrt(d)
    over rows `tokens` of K [L][d] that falls on each logical page in `pages`
    (tokens t with t // ell == page)."""
    q, K = _u16(q), _u16(K)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    pages = np.ascontiguousarray(pages, dtype=np.int32)
    G, d = q.shape
    mass = np.empty((G, pages.size), np.float64)
    qd, kd = _kv(dtype, kv_dtype)
    if lib().orc_page_mass_kv(q, qd, K, kd, float(kscale), G, d, tokens, tokens.size, int(ell),
                              pages, pages.size, mass) != 0:
        raise ValueError("orc_page_mass: empty token set")
    return mass


# ---- prefill: low-rank block importance and block-sparse causal attention ----

def prefill_block_scores(Q, K, dtype, Wq, Wk, blk, kv_dtype=None, kscale=1.0):
    """fp64 [nb][nb] block importance of one kv head (see
    orc_prefill_block_scores): Q [G][L][d], K [L][d], Wq/Wk [d][r] fp32."""
    Q, K = _u16(Q), _u16(K)
    G, L, d = Q.shape
    Wq = np.ascontiguousarray(Wq, np.float32)
    Wk = np.ascontiguousarray(Wk, np.float32)
    r = Wq.shape[1]
    nb = -(-L // blk)
    S = np.empty((nb, nb), np.float64)
    qd, kd = _kv(dtype, kv_dtype)
    if lib().orc_prefill_block_scores(Q, qd, K, kd, float(kscale), Wq, Wk, G, d, r, L, int(blk),
                                      S) != 0:
        raise ValueError("orc_prefill_block_scores: bad arguments")
    return S


def prefill_select(S, blk, L, token_budget, dense_below):
    """Key blocks each query block attends, ascending (LServe write-up,
    section 3.1): below `dense_below` tokens every causal block; otherwise the
    query block's own (diagonal) block plus the best of the earlier ones by
    (score desc, index asc), max(1, token_budget // blk) blocks in all --
    the decode selection rule with the diagonal block in the newest page's
    place."""
    nb = S.shape[0]
    if L < dense_below:
        return [np.arange(b + 1, dtype=np.int32) for b in range(nb)]
    k = max(1, int(token_budget) // int(blk))
    return [select(np.asarray(S[b, :b + 1], np.float32), b + 1, k) for b in range(nb)]


def prefill_attention(Q, K, V, dtype, blocks, blk, kv_dtype=None, kscale=1.0, vscale=1.0):
    """fp64 [G][L][d] causal attention of every query token t over the keys
    s <= t of its query block's chosen key blocks (see orc_prefill_attention;
    per token the two-pass softmax of `attention`)."""
    Q, K, V = _u16(Q), _u16(K), _u16(V)
    G, L, d = Q.shape
    flat = np.ascontiguousarray(np.concatenate([np.asarray(b, np.int32) for b in blocks]),
                                np.int32)
    offs = np.ascontiguousarray(np.cumsum([0] + [len(b) for b in blocks]), np.int32)
    out = np.empty((G, L, d), np.float64)
    qd, kd = _kv(dtype, kv_dtype)
    if lib().orc_prefill_attention(Q, qd, K, V, kd, float(kscale), float(vscale), G, d, L,
                                   int(blk), flat, offs, out) != 0:
        raise ValueError("orc_prefill_attention: bad arguments")
    return out


# ---- decode state on logical positions ------------------------------------

class _Seq:
    def __init__(self, Hkv, d, cap):
        self.L = 0
        self.counter = 0          # decode steps since the sequence started
        self.nL0 = {}             # kv head -> page count when last selected
        self.sel = {}             # kv head -> selected pages (ascending)
        self.K = np.zeros((Hkv, cap, d), np.uint16)
        self.V = np.zeros((Hkv, cap, d), np.uint16)
        self.kmin = {}            # kv head -> [nL][d] bit patterns
        self.kmax = {}


class OracleLayer:
    """One attention layer's KV state and the decode step, on logical positions.

    cfg keys: num_q_heads, num_kv_heads, head_dim, dtype ('f16'/'bf16'),
    logical_page, streaming (list of bool per kv head), sink, window,
    token_budget (<=0: min(4096, L/32)), reuse_interval (C), max_context;
    optional kv_fp8 (K and V stored as fp8 e4m3 codes of value / scale) with
    k_scale, v_scale (per kv head, fp32, default 1).

    Step order (LServe write-up, section 3.2): append the new token, select
    when the sequence's step counter is a multiple of C (or when forced),
    attend, then advance the counter.
    """

    def __init__(self, cfg):
        self.cfg = dict(cfg)
        self.Hq = cfg["num_q_heads"]
        self.Hkv = cfg["num_kv_heads"]
        self.G = self.Hq // self.Hkv
        self.d = cfg["head_dim"]
        self.dtype = dtype_code(cfg["dtype"])
        self.ell = cfg["logical_page"]
        self.streaming = [bool(x) for x in cfg["streaming"]]
        self.S = cfg.get("sink", 0)
        self.W = cfg.get("window", 0)
        self.budget = cfg.get("token_budget", 0)
        self.C = cfg.get("reuse_interval", 4)
        self.cap = cfg["max_context"]
        self.kv_fp8 = bool(cfg.get("kv_fp8", False))
        self.kvdtype = E4M3 if self.kv_fp8 else self.dtype
        one = [1.0] * self.Hkv
        # the scales the GPU path uses are fp32
        self.ks = [float(np.float32(x)) for x in (cfg.get("k_scale") or one)]
        self.vs = [float(np.float32(x)) for x in (cfg.get("v_scale") or one)]
        if not self.kv_fp8:
            self.ks, self.vs = one, one
        self.seqs = {}
        self._next = 0

    def new_seq(self):
        sid = self._next
        self._next += 1
        self.seqs[sid] = _Seq(self.Hkv, self.d, self.cap)
        return sid

    def free_seq(self, sid):
        del self.seqs[sid]

    def dyn_heads(self):
        return [h for h in range(self.Hkv) if not self.streaming[h]]

    # (metadata) ------------------------------------------------------------
    def append(self, sid, k, v):
        """Append tokens k, v [n][Hkv][d] (bit patterns) at positions L..L+n-1
        and recompute the min/max metadata of every logical page they touch."""
        s = self.seqs[sid]
        k, v = _u16(k), _u16(v)
        n = k.shape[0]
        if s.L + n > self.cap:
            raise ValueError("append beyond max_context")
        L0, L1 = s.L, s.L + n
        if self.kv_fp8:  # stored as e4m3 codes of value / scale, per kv head
            for h in range(self.Hkv):
                s.K[h, L0:L1] = quantize_e4m3(k[:, h], self.dtype, self.ks[h])
                s.V[h, L0:L1] = quantize_e4m3(v[:, h], self.dtype, self.vs[h])
        else:
            s.K[:, L0:L1] = k.transpose(1, 0, 2)
            s.V[:, L0:L1] = v.transpose(1, 0, 2)
        s.L = L1
        j0, j1 = L0 // self.ell, -(-L1 // self.ell)
        for h in self.dyn_heads():
            mn, mx = page_minmax(s.K[h, :L1], self.kvdtype, self.ell, j0, j1)
            old_min = s.kmin.get(h, np.zeros((0, self.d), np.uint16))[:j0]
            old_max = s.kmax.get(h, np.zeros((0, self.d), np.uint16))[:j0]
            s.kmin[h] = np.concatenate([old_min, mn])
            s.kmax[h] = np.concatenate([old_max, mx])

    # (score, budget, top-k, reuse) ----------------------------------------
    def selection_due(self, sid):
        return self.seqs[sid].counter % self.C == 0

    def scores(self, sid, q, h):
        s = self.seqs[sid]
        qg = _u16(q)[h * self.G:(h + 1) * self.G]
        return page_scores(qg, s.kmin[h], s.kmax[h], self.dtype, self.kvdtype, self.ks[h])

    def select(self, sid, q, force=False):
        """Run the selection if due (counter % C == 0) or forced; returns
        whether it ran.  Otherwise the stored selection is kept as is."""
        s = self.seqs[sid]
        if not (force or self.selection_due(sid)):
            return False
        if s.L <= 0:
            raise ValueError("select on an empty sequence")
        nL = -(-s.L // self.ell)
        K_sel = budget_pages(s.L, self.budget, self.ell)
        for h in self.dyn_heads():
            S = self.scores(sid, q, h)
            s.sel[h] = select(S, nL, K_sel)
            s.nL0[h] = nL
        return True

    def tokens(self, sid, h):
        """Attended logical positions of kv head h at the current length."""
        s = self.seqs[sid]
        if self.streaming[h]:
            return streaming_tokens(s.L, self.S, self.W)
        return dynamic_tokens(s.sel[h], s.nL0[h], s.L, self.ell)

    # (attention) ------------------------------------------------------------
    def attend(self, sid, q, advance=True, threads=1):
        """Output [Hq][d] fp64 for query q [Hq][d]; advances the step counter."""
        s = self.seqs[sid]
        q = _u16(q)
        out = np.empty((self.Hq, self.d), np.float64)

        def one(h):
            T = self.tokens(sid, h)
            qg = q[h * self.G:(h + 1) * self.G]
            out[h * self.G:(h + 1) * self.G] = attention(
                qg, s.K[h, :s.L], s.V[h, :s.L], self.dtype, T, self.kvdtype, self.ks[h],
                self.vs[h])

        if threads > 1:
            with ThreadPoolExecutor(threads) as ex:
                list(ex.map(one, range(self.Hkv)))
        else:
            for h in range(self.Hkv):
                one(h)
        if advance:
            s.counter += 1
        return out

    def softmax_stats(self, sid, q):
        """(row_max [Hq], row_sum [Hq]) fp64 over each head's attended tokens
        (does not advance the step counter)."""
        s = self.seqs[sid]
        q = _u16(q)
        rm = np.empty(self.Hq, np.float64)
        rs = np.empty(self.Hq, np.float64)
        for h in range(self.Hkv):
            T = self.tokens(sid, h)
            a, b = softmax_stats(q[h * self.G:(h + 1) * self.G], s.K[h, :s.L], self.dtype, T,
                                 self.kvdtype, self.ks[h])
            rm[h * self.G:(h + 1) * self.G] = a
            rs[h * self.G:(h + 1) * self.G] = b
        return rm, rs

    def attended_pages(self, sid, h):
        """Logical pages a dynamic kv head attends, ascending: the stored
        selection plus every page created since it was made."""
        s = self.seqs[sid]
        nL = -(-s.L // self.ell)
        return np.union1d(s.sel[h], np.arange(s.nL0[h] - 1, nL)).astype(np.int32)

    def page_mass(self, sid, q):
        """{dynamic kv head: (pages [n] ascending, mass [G][n] fp64)}: each
        query head's softmax weight per attended logical page (does not
        advance the step counter)."""
        s = self.seqs[sid]
        q = _u16(q)
        res = {}
        for h in self.dyn_heads():
            pages = self.attended_pages(sid, h)
            res[h] = (pages, page_mass(q[h * self.G:(h + 1) * self.G], s.K[h, :s.L], self.dtype,
                                       self.tokens(sid, h), self.ell, pages, self.kvdtype,
                                       self.ks[h]))
        return res

    def step(self, sid, q, k, v, threads=1):
        """One decode step: append one token, select if due, attend."""
        self.append(sid, np.asarray(k)[None], np.asarray(v)[None])
        self.select(sid, q)
        return self.attend(sid, q, threads=threads)


def cpu_threads():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") \
        else os.cpu_count()
