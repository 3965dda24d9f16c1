"""Python binding of the GB300 sparse paged decode attention library.

Thin ctypes marshalling over the C ABI in ``include/spd.h`` (``libspd.so``,
built in-tree by ``build.py``).  Every step of the decode path runs in the
library's CUDA kernels; PyTorch supplies device memory and streams only.
There is no fallback: if ``libspd.so`` is missing, importing the binding
raises.

Low level: ``spd_*`` functions with the C names (config as a dict, device
pointers as ints).  High level: :class:`SparsePagedKVCache`, which allocates
the device buffers with torch and takes torch tensors.
"""
import ctypes
import os

__all__ = ["SpdError", "SparsePagedKVCache", "lib", "LIB_PATH", "make_config"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libspd.so")

SPD_OK = 0
STATUS = {0: "SPD_OK", 1: "SPD_ERR_INVALID_ARG", 2: "SPD_ERR_NO_PAGES",
          3: "SPD_ERR_BAD_SEQ", 4: "SPD_ERR_CAPACITY", 5: "SPD_ERR_CUDA",
          6: "SPD_ERR_DEVICE_CHECK", 7: "SPD_ERR_STATE"}
DTYPES = {"f16": 0, "fp16": 0, "float16": 0, "bf16": 1, "bfloat16": 1}
BUFFER_FIELDS = ("k_pool", "v_pool", "meta", "stream_k", "stream_v",
                 "page_table", "selection", "scratch")


class SpdError(RuntimeError):
    def __init__(self, status, where, detail=""):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__("%s: %s%s" % (where, self.name,
                                       (" (" + detail + ")") if detail else ""))


class spd_config(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int),
                ("logical_page", ctypes.c_int), ("physical_page", ctypes.c_int),
                ("num_physical_pages", ctypes.c_int), ("max_seqs", ctypes.c_int),
                ("max_context", ctypes.c_int),
                ("kv_head_is_streaming", ctypes.POINTER(ctypes.c_ubyte)),
                ("sink", ctypes.c_int), ("window", ctypes.c_int),
                ("token_budget", ctypes.c_int), ("reuse_interval", ctypes.c_int),
                ("free_list_seed", ctypes.c_ulonglong), ("kv_fp8", ctypes.c_int),
                ("k_scale", ctypes.POINTER(ctypes.c_float)),
                ("v_scale", ctypes.POINTER(ctypes.c_float))]


class spd_prefill_config(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int), ("rank", ctypes.c_int),
                ("block", ctypes.c_int), ("token_budget", ctypes.c_int),
                ("dense_below", ctypes.c_int)]


class spd_sizes(ctypes.Structure):
    _fields_ = [(f, ctypes.c_size_t) for f in BUFFER_FIELDS]


class spd_buffers(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in BUFFER_FIELDS]


_lib = None


def lib():
    """The loaded ``libspd.so``; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("libspd.so is not built (run __graft_entry__.build() "
                          "or python sparse_paged_decode_logical_gb300/build.py)")
    L = ctypes.CDLL(LIB_PATH)
    vp, ip, i, st = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int), ctypes.c_int, ctypes.c_int
    ll = ctypes.POINTER(ctypes.c_longlong)
    sig = {
        "spd_query_sizes": [ctypes.POINTER(spd_config), ctypes.POINTER(spd_sizes)],
        "spd_create": [ctypes.POINTER(spd_config), ctypes.POINTER(spd_buffers),
                       ctypes.POINTER(vp)],
        "spd_seq_create": [vp, ip],
        "spd_seq_free": [vp, i],
        "spd_seq_reserve": [vp, i, i],
        "spd_seq_info": [vp, i, ll, ll, ip, ip],
        "spd_get_page_table": [vp, i, ip, i, ip],
        "spd_free_pages": [vp, ip],
        "spd_kv_append": [vp, ip, i, i, vp, vp, vp],
        "spd_select_pages": [vp, vp, ip, i, i, vp],
        "spd_sparse_decode_attention": [vp, vp, ip, i, vp, vp],
        "spd_sparse_decode_attention_static": [vp, vp, ip, i, vp, vp],
        "spd_sparse_decode_attention_stats": [vp, vp, ip, i, vp, vp, vp, vp],
        "spd_sparse_decode_attention_page_mass": [vp, vp, ip, i, vp, vp, vp, vp, vp, i, vp],
        "spd_decode_step": [vp, vp, vp, vp, ip, i, vp, vp],
        "spd_get_selection": [vp, i, i, ip, i, ip, vp],
        "spd_check_status": [vp, vp],
        "spd_launch_count": [vp, ll],
        "spd_set_early_kv_staging": [vp, i],
        "spd_prefill_sizes": [ctypes.POINTER(spd_prefill_config), i, ip,
                              ctypes.POINTER(ctypes.c_size_t)],
        "spd_prefill_block_sparse_attention": [ctypes.POINTER(spd_prefill_config), i, vp, vp, vp,
                                               vp, vp, vp, vp, vp, ctypes.c_size_t, vp],
        "spd_prefill_check": [vp, vp],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = st
    L.spd_destroy.argtypes = [vp]
    L.spd_destroy.restype = None
    L.spd_status_string.argtypes = [st]
    L.spd_status_string.restype = ctypes.c_char_p
    L.spd_last_error.argtypes = [vp]
    L.spd_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


# ---- low level: the C entry points with Python arguments --------------------

def make_config(num_q_heads, num_kv_heads, head_dim, dtype, logical_page,
                physical_page, num_physical_pages, max_seqs, max_context,
                streaming=None, sink=0, window=0, token_budget=0,
                reuse_interval=4, free_list_seed=0, kv_fp8=False, k_scale=None,
                v_scale=None):
    """Build an ``spd_config`` (the streaming mask and scale arrays are kept
    alive on it).  kv_fp8: store K/V as fp8 E4M3 codes of value / scale, with
    per-kv-head k_scale / v_scale (default 1)."""
    c = spd_config()
    c.num_q_heads, c.num_kv_heads, c.head_dim = num_q_heads, num_kv_heads, head_dim
    c.dtype = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    c.logical_page, c.physical_page = logical_page, physical_page
    c.num_physical_pages, c.max_seqs, c.max_context = num_physical_pages, max_seqs, max_context
    if streaming is not None:
        arr = (ctypes.c_ubyte * num_kv_heads)(*[1 if s else 0 for s in streaming])
        c._streaming = arr
        c.kv_head_is_streaming = ctypes.cast(arr, ctypes.POINTER(ctypes.c_ubyte))
    c.sink, c.window, c.token_budget = sink, window, token_budget
    c.reuse_interval, c.free_list_seed = reuse_interval, free_list_seed
    c.kv_fp8 = 1 if kv_fp8 else 0
    for name, vals in (("k_scale", k_scale), ("v_scale", v_scale)):
        if vals is not None:
            arr = (ctypes.c_float * num_kv_heads)(*[float(x) for x in vals])
            setattr(c, "_" + name, arr)
            setattr(c, name, ctypes.cast(arr, ctypes.POINTER(ctypes.c_float)))
    return c


def _check(st, where, ctx=None):
    if st != SPD_OK:
        detail = ""
        if ctx:
            detail = (lib().spd_last_error(ctx) or b"").decode()
        raise SpdError(st, where, detail)


def _ids(seq_ids):
    seq_ids = [int(s) for s in seq_ids]
    return (ctypes.c_int * len(seq_ids))(*seq_ids), len(seq_ids)


def spd_query_sizes(cfg):
    out = spd_sizes()
    _check(lib().spd_query_sizes(ctypes.byref(cfg), ctypes.byref(out)), "spd_query_sizes")
    return {f: getattr(out, f) for f in BUFFER_FIELDS}


def spd_create(cfg, buffers):
    """buffers: dict field -> device address (int)."""
    b = spd_buffers(*[buffers.get(f) or None for f in BUFFER_FIELDS])
    ctx = ctypes.c_void_p()
    _check(lib().spd_create(ctypes.byref(cfg), ctypes.byref(b), ctypes.byref(ctx)),
           "spd_create")
    return ctx


def spd_destroy(ctx):
    lib().spd_destroy(ctx)


def spd_seq_create(ctx):
    sid = ctypes.c_int()
    _check(lib().spd_seq_create(ctx, ctypes.byref(sid)), "spd_seq_create", ctx)
    return sid.value


def spd_seq_free(ctx, seq_id):
    _check(lib().spd_seq_free(ctx, int(seq_id)), "spd_seq_free", ctx)


def spd_seq_reserve(ctx, seq_id, n_tokens):
    _check(lib().spd_seq_reserve(ctx, int(seq_id), int(n_tokens)), "spd_seq_reserve", ctx)


def spd_seq_info(ctx, seq_id):
    L, cnt = ctypes.c_longlong(), ctypes.c_longlong()
    nl0, kept = ctypes.c_int(), ctypes.c_int()
    _check(lib().spd_seq_info(ctx, int(seq_id), ctypes.byref(L), ctypes.byref(cnt),
                              ctypes.byref(nl0), ctypes.byref(kept)), "spd_seq_info", ctx)
    return dict(length=L.value, step_counter=cnt.value,
                pages_at_selection=nl0.value, pages_kept=kept.value)


def spd_get_page_table(ctx, seq_id):
    n = ctypes.c_int()
    _check(lib().spd_get_page_table(ctx, int(seq_id), None, 0, ctypes.byref(n)),
           "spd_get_page_table", ctx)
    arr = (ctypes.c_int * max(n.value, 1))()
    _check(lib().spd_get_page_table(ctx, int(seq_id), arr, n.value, ctypes.byref(n)),
           "spd_get_page_table", ctx)
    return list(arr[:n.value])


def spd_free_pages(ctx):
    n = ctypes.c_int()
    _check(lib().spd_free_pages(ctx, ctypes.byref(n)), "spd_free_pages", ctx)
    return n.value


def spd_kv_append(ctx, seq_ids, n_tokens, k_ptr, v_ptr, stream=0):
    ids, n = _ids(seq_ids)
    _check(lib().spd_kv_append(ctx, ids, n, int(n_tokens), k_ptr, v_ptr, stream or None),
           "spd_kv_append", ctx)


def spd_select_pages(ctx, q_ptr, seq_ids, force=False, stream=0):
    ids, n = _ids(seq_ids)
    _check(lib().spd_select_pages(ctx, q_ptr, ids, n, 1 if force else 0, stream or None),
           "spd_select_pages", ctx)


def spd_sparse_decode_attention(ctx, q_ptr, seq_ids, out_ptr, stream=0):
    ids, n = _ids(seq_ids)
    _check(lib().spd_sparse_decode_attention(ctx, q_ptr, ids, n, out_ptr, stream or None),
           "spd_sparse_decode_attention", ctx)


def spd_sparse_decode_attention_static(ctx, q_ptr, seq_ids, out_ptr, stream=0):
    """spd_sparse_decode_attention with its temporaries in the library-owned
    device array: for callers that cannot allocate device memory at call
    time (see include/spd.h)."""
    ids, n = _ids(seq_ids)
    _check(lib().spd_sparse_decode_attention_static(ctx, q_ptr, ids, n, out_ptr, stream or None),
           "spd_sparse_decode_attention_static", ctx)


def spd_sparse_decode_attention_stats(ctx, q_ptr, seq_ids, out_ptr, row_max_ptr, row_sum_ptr,
                                      stream=0):
    ids, n = _ids(seq_ids)
    _check(lib().spd_sparse_decode_attention_stats(ctx, q_ptr, ids, n, out_ptr, row_max_ptr,
                                                   row_sum_ptr, stream or None),
           "spd_sparse_decode_attention_stats", ctx)


def spd_sparse_decode_attention_page_mass(ctx, q_ptr, seq_ids, out_ptr, row_max_ptr, row_sum_ptr,
                                          pages_ptr, mass_ptr, max_pages, stream=0):
    ids, n = _ids(seq_ids)
    _check(lib().spd_sparse_decode_attention_page_mass(ctx, q_ptr, ids, n, out_ptr,
                                                       row_max_ptr or None, row_sum_ptr or None,
                                                       pages_ptr or None, mass_ptr or None,
                                                       max_pages, stream or None),
           "spd_sparse_decode_attention_page_mass", ctx)


def spd_decode_step(ctx, q_ptr, k_ptr, v_ptr, seq_ids, out_ptr, stream=0):
    ids, n = _ids(seq_ids)
    _check(lib().spd_decode_step(ctx, q_ptr, k_ptr, v_ptr, ids, n, out_ptr, stream or None),
           "spd_decode_step", ctx)


def spd_get_selection(ctx, seq_id, kv_head, stream=0):
    n = ctypes.c_int()
    _check(lib().spd_get_selection(ctx, int(seq_id), int(kv_head), None, 0,
                                   ctypes.byref(n), stream or None), "spd_get_selection", ctx)
    arr = (ctypes.c_int * max(n.value, 1))()
    _check(lib().spd_get_selection(ctx, int(seq_id), int(kv_head), arr, n.value,
                                   ctypes.byref(n), stream or None), "spd_get_selection", ctx)
    return list(arr[:n.value])


def spd_check_status(ctx, stream=0):
    _check(lib().spd_check_status(ctx, stream or None), "spd_check_status", ctx)


def spd_set_early_kv_staging(ctx, enable):
    _check(lib().spd_set_early_kv_staging(ctx, 1 if enable else 0), "spd_set_early_kv_staging", ctx)


def spd_launch_count(ctx):
    n = ctypes.c_longlong()
    _check(lib().spd_launch_count(ctx, ctypes.byref(n)), "spd_launch_count", ctx)
    return n.value


# ---- high level: torch-allocated buffers ----------------------------------------

class SparsePagedKVCache:
    """One attention layer's paged KV cache on a CUDA device.

    Buffers come from ``torch.empty`` on ``device``; all calls enqueue on the
    current torch stream of that device unless ``stream`` is given.
    """

    def __init__(self, device="cuda", **cfg):
        import torch
        self.torch = torch
        self.cfg_dict = dict(cfg)
        self.cfg = make_config(**cfg)
        dev = torch.device(device)
        if dev.type == "cuda" and dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        self.sizes = spd_query_sizes(self.cfg)
        self.buffers = {}
        addrs = {}
        for f in BUFFER_FIELDS:
            n = self.sizes[f]
            if n:
                t = torch.empty(n, dtype=torch.uint8, device=self.device)
                self.buffers[f] = t
                addrs[f] = t.data_ptr()
        self.ctx = spd_create(self.cfg, addrs)
        self.Hq, self.Hkv, self.d = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
        self.dtype = torch.bfloat16 if DTYPES[cfg["dtype"]] == 1 else torch.float16
        # per-call marshalling state: the device index as an int, the raw
        # current-stream query, ctypes id arrays by id tuple, the entry point
        self._dev_index = self.device.index
        self._raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        self._ids_cache = {}
        self._step_fn = lib().spd_decode_step

    def __del__(self):
        ctx = getattr(self, "ctx", None)
        if ctx:
            spd_destroy(ctx)
            self.ctx = None

    def _stream(self, stream):
        if stream is None:
            if self._raw_stream is not None:
                return self._raw_stream(self._dev_index)
            stream = self.torch.cuda.current_stream(self.device)
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)

    def _ptr(self, t, shape, dtype):
        if t.shape != shape or t.dtype != dtype or not t.is_contiguous() \
                or t.get_device() != self._dev_index:
            raise ValueError("expected contiguous %s tensor %s on %s, got %s %s on %s"
                             % (dtype, tuple(shape), self.device, t.dtype, tuple(t.shape),
                                t.device))
        return t.data_ptr()

    def seq_create(self):
        return spd_seq_create(self.ctx)

    def seq_free(self, seq_id):
        spd_seq_free(self.ctx, seq_id)

    def seq_reserve(self, seq_id, n_tokens):
        spd_seq_reserve(self.ctx, seq_id, n_tokens)

    def seq_info(self, seq_id):
        return spd_seq_info(self.ctx, seq_id)

    def page_table(self, seq_id):
        return spd_get_page_table(self.ctx, seq_id)

    def free_pages(self):
        return spd_free_pages(self.ctx)

    def kv_append(self, seq_ids, k, v, stream=None):
        """k, v: [n_seqs][n_tokens][Hkv][d] of the cache dtype."""
        n = len(seq_ids)
        shape = (n, k.shape[1], self.Hkv, self.d)
        spd_kv_append(self.ctx, seq_ids, k.shape[1], self._ptr(k, shape, self.dtype),
                      self._ptr(v, shape, self.dtype), self._stream(stream))

    def select_pages(self, q, seq_ids, force=False, stream=None):
        qp = self._ptr(q, (len(seq_ids), self.Hq, self.d), self.dtype)
        spd_select_pages(self.ctx, qp, seq_ids, force, self._stream(stream))

    def sparse_decode_attention(self, q, seq_ids, out=None, stream=None):
        n = len(seq_ids)
        qp = self._ptr(q, (n, self.Hq, self.d), self.dtype)
        if out is None:
            out = self.torch.empty((n, self.Hq, self.d), dtype=self.torch.float32,
                                   device=self.device)
        op = self._ptr(out, (n, self.Hq, self.d), self.torch.float32)
        spd_sparse_decode_attention(self.ctx, qp, seq_ids, op, self._stream(stream))
        return out

    def sparse_decode_attention_stats(self, q, seq_ids, stream=None):
        """Attention plus the per-head softmax statistics: returns (out,
        row_max, row_sum) with row_max = max logit, row_sum = sum of
        exp(logit - row_max) over the attended tokens, [n][Hq] fp32."""
        n = len(seq_ids)
        qp = self._ptr(q, (n, self.Hq, self.d), self.dtype)
        out = self.torch.empty((n, self.Hq, self.d), dtype=self.torch.float32, device=self.device)
        rm = self.torch.empty((n, self.Hq), dtype=self.torch.float32, device=self.device)
        rs = self.torch.empty((n, self.Hq), dtype=self.torch.float32, device=self.device)
        spd_sparse_decode_attention_stats(self.ctx, qp, seq_ids,
                                          self._ptr(out, (n, self.Hq, self.d), self.torch.float32),
                                          self._ptr(rm, (n, self.Hq), self.torch.float32),
                                          self._ptr(rs, (n, self.Hq), self.torch.float32),
                                          self._stream(stream))
        return out, rm, rs

    def attended_page_count(self, seq_id):
        """Logical pages each dynamic head of the sequence attends now: the
        stored selection plus the pages created since it was taken."""
        info = self.seq_info(seq_id)
        ell = self.cfg_dict["logical_page"]
        return info["pages_kept"] + -(-info["length"] // ell) - info["pages_at_selection"]

    def sparse_decode_attention_page_mass(self, q, seq_ids, max_pages=None, stream=None):
        """Attention, the softmax statistics and the per-page attention mass of
        the dynamic heads: returns (out [n][Hq][d], row_max [n][Hq], row_sum
        [n][Hq], pages [n][Hd][max_pages] int32 (-1 padded), mass
        [n][Hd][G][max_pages] fp32).  max_pages defaults to the largest
        attended page count among the sequences."""
        n = len(seq_ids)
        Hd = sum(1 for x in (self.cfg_dict.get("streaming") or [False] * self.Hkv) if not x)
        G = self.Hq // self.Hkv
        if max_pages is None:
            max_pages = max([self.attended_page_count(s) for s in seq_ids] + [1]) if Hd else 1
        qp = self._ptr(q, (n, self.Hq, self.d), self.dtype)
        t, f32 = self.torch, self.torch.float32
        out = t.empty((n, self.Hq, self.d), dtype=f32, device=self.device)
        rm = t.empty((n, self.Hq), dtype=f32, device=self.device)
        rs = t.empty((n, self.Hq), dtype=f32, device=self.device)
        pages = t.empty((n, Hd, max_pages), dtype=t.int32, device=self.device)
        mass = t.empty((n, Hd, G, max_pages), dtype=f32, device=self.device)
        spd_sparse_decode_attention_page_mass(
            self.ctx, qp, seq_ids, self._ptr(out, (n, self.Hq, self.d), f32),
            self._ptr(rm, (n, self.Hq), f32), self._ptr(rs, (n, self.Hq), f32),
            pages.data_ptr() if Hd else 0, mass.data_ptr() if Hd else 0, max_pages,
            self._stream(stream))
        return out, rm, rs, pages, mass

    def decode_step(self, q, k, v, seq_ids, out=None, stream=None):
        key = tuple(seq_ids)
        ids = self._ids_cache.get(key)
        if ids is None:
            ids = _ids(key)
            if len(self._ids_cache) < 1024:
                self._ids_cache[key] = ids
        n = ids[1]
        qp = self._ptr(q, (n, self.Hq, self.d), self.dtype)
        kp = self._ptr(k, (n, self.Hkv, self.d), self.dtype)
        vp = self._ptr(v, (n, self.Hkv, self.d), self.dtype)
        if out is None:
            out = self.torch.empty((n, self.Hq, self.d), dtype=self.torch.float32,
                                   device=self.device)
        op = self._ptr(out, (n, self.Hq, self.d), self.torch.float32)
        st = self._step_fn(self.ctx, qp, kp, vp, ids[0], n, op, self._stream(stream) or None)
        if st != SPD_OK:
            _check(st, "spd_decode_step", self.ctx)
        return out

    def selection(self, seq_id, kv_head, stream=None):
        return spd_get_selection(self.ctx, seq_id, kv_head, self._stream(stream))

    def check_status(self, stream=None):
        spd_check_status(self.ctx, self._stream(stream))

    def launch_count(self):
        return spd_launch_count(self.ctx)

    def set_early_kv_staging(self, enable=True):
        spd_set_early_kv_staging(self.ctx, enable)


# ---- prefill: block-sparse attention of one prompt ----------------------------

def prefill_block_sparse_attention(q, k, v, w_q, w_k, block=64, token_budget=4096,
                                   dense_below=32768, stream=None, check=True):
    """Block-sparse causal attention of a prompt (spd_prefill_block_sparse_attention).

    q [L][Hq][d], k, v [L][Hkv][d] (fp16 or bf16, one CUDA device), w_q, w_k
    fp32 [Hkv][d][r].  Returns (out fp32 [L][Hq][d], blocks int32
    [Hkv][nb][KB]: the key blocks each query block attended, -1 padded)."""
    import torch
    L, Hq, d = q.shape
    Hkv = k.shape[1]
    r = w_q.shape[2]
    dt = q.dtype
    if dt not in (torch.float16, torch.bfloat16) or k.dtype != dt or v.dtype != dt:
        raise ValueError("q, k, v must share one dtype, fp16 or bf16")
    for t, shape in ((k, (L, Hkv, d)), (v, (L, Hkv, d)), (w_q, (Hkv, d, r)), (w_k, (Hkv, d, r))):
        if tuple(t.shape) != shape or not t.is_contiguous() or t.device != q.device:
            raise ValueError("expected a contiguous tensor %s on %s" % (shape, q.device))
    if w_q.dtype != torch.float32 or w_k.dtype != torch.float32 or not q.is_contiguous():
        raise ValueError("w_q, w_k must be fp32 and q contiguous")
    cfg = spd_prefill_config(Hq, Hkv, d, 1 if dt == torch.bfloat16 else 0, r, block,
                             token_budget, dense_below)
    kb, ws = ctypes.c_int(), ctypes.c_size_t()
    _check(lib().spd_prefill_sizes(ctypes.byref(cfg), L, ctypes.byref(kb), ctypes.byref(ws)),
           "spd_prefill_sizes")
    nb = -(-L // block)
    out = torch.empty((L, Hq, d), dtype=torch.float32, device=q.device)
    blocks = torch.empty((Hkv, nb, kb.value), dtype=torch.int32, device=q.device)
    work = torch.empty(ws.value, dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _check(lib().spd_prefill_block_sparse_attention(
        ctypes.byref(cfg), L, q.data_ptr(), k.data_ptr(), v.data_ptr(), w_q.data_ptr(),
        w_k.data_ptr(), out.data_ptr(), blocks.data_ptr(), work.data_ptr(), ws.value,
        st or None), "spd_prefill_block_sparse_attention")
    if check:
        _check(lib().spd_prefill_check(work.data_ptr(), st or None), "spd_prefill_check")
    return out, blocks
