"""Seeded synthetic inputs for sparse paged decode attention.

This module holds no part of the method's arithmetic.  It only draws the
random keys, values and queries that both the CUDA library and the oracle
consume, with the shapes and structure of the workloads the LServe write-up
and its companions measure on (Llama-3-8B and Llama-2-7B attention layers at
32K-256K context, 4K token budget, reuse interval C = 4):

* K, V ~ N(0, 1) in fp32, rounded to nearest even into fp16 / bf16;
* outlier channels: two seeded channel indices of every key scaled x50
  (the massive-activation channels of the Novita KV-sparsity article);
* planted needles: keys k = 4 * qbar_g / |qbar_g| where qbar_g is the mean
  query base vector of the kv head's query group, either at a fraction of
  token positions or as whole logical pages at fixed depths;
* queries: a base vector u ~ N(0, I) per (sequence, query head); at decode
  step s the query is u + 0.25 * eps_s.

Seeds: numpy.random.default_rng([20260 + config_index, layer, stream, ...]).
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np


@dataclass
class Workload:
    name: str
    index: int                 # 0..4, also the seed offset
    batch: int
    Hq: int
    Hkv: int
    d: int
    context: int               # tokens already in the cache before decode
    ell: int                   # logical page (selection unit)
    P: int                     # physical page (allocation unit)
    dtype: str                 # 'f16' | 'bf16'
    streaming: List[bool]      # per kv head
    sink: int
    window: int
    token_budget: int          # <= 0: min(4096, L/32)
    C: int
    steps: int
    needle: str                # 'none' | 'tokens' | 'pages'
    needle_frac: float = 0.0
    needle_depths: tuple = ()
    outliers: bool = False
    permute_pages: bool = False
    log_uniform_lens: Optional[tuple] = None   # (lo, hi) for mixed batches
    notes: str = ""
    lens: List[int] = field(default_factory=list)

    @property
    def G(self):
        return self.Hq // self.Hkv

    def seq_lens(self):
        if self.lens:
            return list(self.lens)
        if self.log_uniform_lens is None:
            return [self.context] * self.batch
        lo, hi = self.log_uniform_lens
        r = np.random.default_rng([20260 + self.index, 7777])
        u = r.uniform(np.log(lo), np.log(hi), size=self.batch)
        return [int(round(float(np.exp(x)))) for x in u]

    def max_context(self):
        return max(self.seq_lens()) + self.steps + 64

    def lib_config(self, num_physical_pages=None, free_list_seed=None):
        """Keyword arguments for the library/oracle configuration."""
        lens = self.seq_lens()
        mc = self.max_context()
        if num_physical_pages is None:
            num_physical_pages = sum(-(-(L + self.steps + 64) // self.P) for L in lens)
        if free_list_seed is None:
            free_list_seed = (1000 + self.index) if self.permute_pages else 0
        return dict(num_q_heads=self.Hq, num_kv_heads=self.Hkv, head_dim=self.d,
                    dtype=self.dtype, logical_page=self.ell, physical_page=self.P,
                    num_physical_pages=num_physical_pages, max_seqs=self.batch,
                    max_context=mc, streaming=list(self.streaming),
                    sink=self.sink, window=self.window,
                    token_budget=self.token_budget, reuse_interval=self.C,
                    free_list_seed=free_list_seed)


def _half(n, Hkv):
    return [h < n for h in range(Hkv)]


# The five workloads (shapes, structure, steps) -------------------------------
WORKLOADS = {
    "tiny": Workload(
        name="tiny", index=0, batch=1, Hq=4, Hkv=2, d=64, context=4096, ell=16,
        P=64, dtype="f16", streaming=[False, True], sink=16, window=256,
        token_budget=512, C=4, steps=8, needle="tokens", needle_frac=0.01,
        notes="kv head 0 dynamic (budget 512), kv head 1 streaming (16+256)"),
    "llama3_8b_b4_32k": Workload(
        name="llama3_8b_b4_32k", index=1, batch=4, Hq=32, Hkv=8, d=128,
        context=32768, ell=32, P=512, dtype="f16", streaming=_half(4, 8),
        sink=128, window=2048, token_budget=4096, C=4, steps=16,
        needle="tokens", needle_frac=0.005, outliers=True, permute_pages=True),
    "llama3_8b_b1_128k": Workload(
        name="llama3_8b_b1_128k", index=2, batch=1, Hq=32, Hkv=8, d=128,
        context=131072, ell=32, P=1024, dtype="bf16", streaming=_half(4, 8),
        sink=128, window=4096, token_budget=0, C=4, steps=32,
        needle="pages", needle_depths=(0.1, 0.5, 0.9)),
    "llama2_7b_mha_256k": Workload(
        name="llama2_7b_mha_256k", index=3, batch=1, Hq=32, Hkv=32, d=128,
        context=262144, ell=64, P=1024, dtype="f16", streaming=_half(16, 32),
        sink=64, window=1024, token_budget=4096, C=4, steps=16,
        needle="tokens", needle_frac=0.005),
    "cont_batch_16": Workload(
        name="cont_batch_16", index=4, batch=16, Hq=32, Hkv=8, d=128,
        context=0, ell=32, P=512, dtype="bf16", streaming=[False] * 8, sink=0,
        window=0, token_budget=0, C=4, steps=64, needle="none", outliers=True,
        permute_pages=True, log_uniform_lens=(8192, 131072)),
}


def workload(name, **overrides):
    import dataclasses
    return dataclasses.replace(WORKLOADS[name], **overrides)


# ---- rounding of fp32 draws into the 16-bit storage formats ---------------

def to_bits(x, dtype):
    """fp32 array -> uint16 bit patterns, round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype in ("f16", "fp16", "float16"):
        with np.errstate(over="ignore"):
            return x.astype(np.float16).view(np.uint16)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = 0x7FC0
    return r


# ---- draws ---------------------------------------------------------------

def _rng(wl, *stream):
    return np.random.default_rng([20260 + wl.index] + [int(s) for s in stream])


def outlier_channels(wl, layer=0):
    if not wl.outliers:
        return np.zeros(0, np.int64)
    return np.sort(_rng(wl, layer, 1).choice(wl.d, size=2, replace=False))


def query_base(wl, layer=0):
    """u [B][Hq][d] fp32."""
    return _rng(wl, layer, 2).standard_normal((wl.batch, wl.Hq, wl.d),
                                              dtype=np.float32)


def needle_keys(wl, layer=0):
    """[B][Hkv][d] fp32: 4 * qbar / |qbar| per kv head's query group."""
    u = query_base(wl, layer)
    qbar = u.reshape(wl.batch, wl.Hkv, wl.G, wl.d).mean(axis=2)
    nrm = np.linalg.norm(qbar, axis=-1, keepdims=True)
    return (4.0 * qbar / nrm).astype(np.float32)


def needle_mask(wl, seq, L, layer=0):
    """bool [L]: positions that carry a planted needle key."""
    m = np.zeros(L, bool)
    if wl.needle == "tokens" and wl.needle_frac > 0:
        n = max(1, int(round(wl.needle_frac * L)))
        pos = _rng(wl, layer, 3, seq).choice(L, size=min(n, L), replace=False)
        m[pos] = True
    elif wl.needle == "pages":
        for frac in wl.needle_depths:
            j = int(frac * (L // wl.ell))
            m[j * wl.ell:min((j + 1) * wl.ell, L)] = True
    return m


def context(wl, seq, L=None, layer=0):
    """Context keys/values of one sequence: (K, V) uint16 [L][Hkv][d]."""
    lens = wl.seq_lens()
    L = lens[seq] if L is None else L
    r = _rng(wl, layer, 4, seq)
    K = r.standard_normal((L, wl.Hkv, wl.d), dtype=np.float32)
    V = r.standard_normal((L, wl.Hkv, wl.d), dtype=np.float32)
    m = needle_mask(wl, seq, L, layer)
    if m.any():
        K[m] = needle_keys(wl, layer)[seq][None]
    ch = outlier_channels(wl, layer)
    if ch.size:
        K[:, :, ch] *= 50.0
    return to_bits(K, wl.dtype), to_bits(V, wl.dtype)


def step_tokens(wl, step, layer=0):
    """Decode step inputs: q [B][Hq][d], k, v [B][Hkv][d] (uint16 bits)."""
    r = _rng(wl, layer, 5, step)
    u = query_base(wl, layer)
    q = u + 0.25 * r.standard_normal(u.shape, dtype=np.float32)
    k = r.standard_normal((wl.batch, wl.Hkv, wl.d), dtype=np.float32)
    v = r.standard_normal((wl.batch, wl.Hkv, wl.d), dtype=np.float32)
    ch = outlier_channels(wl, layer)
    if ch.size:
        k[:, :, ch] *= 50.0
    return to_bits(q, wl.dtype), to_bits(k, wl.dtype), to_bits(v, wl.dtype)


def device_context(wl, seq, L, layer, device, generator_seed=None):
    """Same distribution as ``context`` drawn on the GPU with torch's
    generator (used only where the oracle does not read the data, e.g. the
    benchmark's extra layer instances).  Returns (K, V) torch tensors
    [L][Hkv][d] of the workload dtype."""
    import torch
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
    g = torch.Generator(device=device)
    g.manual_seed(generator_seed if generator_seed is not None
                  else (20260 + wl.index) * 1000003 + layer * 1009 + seq)
    K = torch.randn((L, wl.Hkv, wl.d), generator=g, device=device,
                    dtype=torch.float32)
    V = torch.randn((L, wl.Hkv, wl.d), generator=g, device=device,
                    dtype=torch.float32)
    m = torch.from_numpy(needle_mask(wl, seq, L, layer)).to(device)
    if bool(m.any()):
        nk = torch.from_numpy(needle_keys(wl, layer)[seq]).to(device)
        K[m] = nk[None]
    ch = outlier_channels(wl, layer)
    if ch.size:
        K[:, :, torch.from_numpy(ch).to(device)] *= 50.0
    return K.to(tdt), V.to(tdt)
