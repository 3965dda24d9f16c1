"""Drives the CUDA library (through the C ABI binding) and the CPU oracle on
the same seeded inputs and compares them.  Test infrastructure.

Acceptance (restating the target's tolerances):
  * page table, K/V placement and min/max metadata: bit-exact (+0 == -0),
    fp8 storage included (the codes of value / scale);
  * selected page sets: identical, except pages whose oracle score lies
    within 1e-4 * max(|S_cut|, 1e-30) of the cut score S_cut;
  * attention: max |gpu - oracle| <= 2e-3 and mean <= 2e-4, the oracle run
    on the GPU's own selection (so a boundary tie cannot masquerade as an
    attention error), and on its own selection when the sets agree.
"""
import numpy as np
import torch

import oracle
import workloads as W
import sparse_paged_decode_logical_gb300 as spd

TOL_MAX = 2e-3
TOL_MEAN = 2e-4
BAND = 1e-4


def tdev(bits, dtype, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16).to(device)


def bits_equal(a, b, magnitude=0x7FFF):
    """Equal bit patterns, +0 and -0 counted equal (magnitude: the bits below
    the sign: 0x7FFF for 16-bit floats, 0x7F for fp8 codes)."""
    a = np.asarray(a, np.uint16)
    b = np.asarray(b, np.uint16)
    same = a == b
    zero = ((a & magnitude) == 0) & ((b & magnitude) == 0)
    return bool(np.all(same | zero))


def oracle_cfg(cfg):
    return dict(num_q_heads=cfg["num_q_heads"], num_kv_heads=cfg["num_kv_heads"],
                head_dim=cfg["head_dim"], dtype=cfg["dtype"],
                logical_page=cfg["logical_page"], streaming=cfg["streaming"],
                sink=cfg["sink"], window=cfg["window"],
                token_budget=cfg["token_budget"], reuse_interval=cfg["reuse_interval"],
                max_context=cfg["max_context"], kv_fp8=cfg.get("kv_fp8", False),
                k_scale=cfg.get("k_scale"), v_scale=cfg.get("v_scale"))


class Pair:
    """A GPU cache and an oracle layer fed identically."""

    def __init__(self, wl, layer=0, device="cuda", cfg_overrides=None, prefill=True):
        self.wl = wl
        self.layer = layer
        self.lens = wl.seq_lens()
        cfg = wl.lib_config()
        cfg.update(cfg_overrides or {})
        self.cfg = cfg
        self.dt = cfg["dtype"]
        self.cache = spd.SparsePagedKVCache(device=device, **cfg)
        self.orc = oracle.OracleLayer(oracle_cfg(cfg))
        self.device = device
        self.gids, self.oids = [], []
        self.dyn = [h for h in range(cfg["num_kv_heads"]) if not cfg["streaming"][h]]
        self.strm = [h for h in range(cfg["num_kv_heads"]) if cfg["streaming"][h]]
        for b in range(wl.batch):
            self.gids.append(self.cache.seq_create())
            self.oids.append(self.orc.new_seq())
        if prefill:
            for b in range(wl.batch):
                if self.lens[b] > 0:
                    K, V = W.context(wl, b, self.lens[b], layer)
                    self.append_seq(b, K, V)
        self.records = []

    def append_seq(self, b, K, V):
        """K, V [n][Hkv][d] bits for sequence b."""
        self.cache.kv_append([self.gids[b]], tdev(K, self.dt, self.device)[None],
                             tdev(V, self.dt, self.device)[None])
        self.orc.append(self.oids[b], K, V)

    # ---- comparisons ---------------------------------------------------------
    def check_layout(self):
        """Page table, pool rows, streaming slots and metadata vs the oracle."""
        cfg, c = self.cfg, self.cache
        torch.cuda.synchronize()
        d, P, ell = cfg["head_dim"], cfg["physical_page"], cfg["logical_page"]
        R = P // ell
        Hd, Hs = len(self.dyn), len(self.strm)
        N = cfg["num_physical_pages"]
        S, Wn = cfg["sink"], cfg["window"]
        fp8 = bool(cfg.get("kv_fp8"))
        mag = 0x7F if fp8 else 0x7FFF

        def elems(name):  # stored elements: fp8 codes (bytes) or 16-bit patterns
            t = c.buffers[name]
            return t.cpu().numpy() if fp8 else t.view(torch.int16).cpu().numpy().view(np.uint16)

        if Hd:
            kp, vp = elems("k_pool"), elems("v_pool")
            kp, vp = kp.reshape(N, Hd, P, d), vp.reshape(N, Hd, P, d)
            meta = elems("meta").reshape(N, Hd, R, 2, d)
        if Hs:
            sk, sv = elems("stream_k"), elems("stream_v")
            sk = sk.reshape(cfg["max_seqs"], Hs, S + Wn, d)
            sv = sv.reshape(cfg["max_seqs"], Hs, S + Wn, d)
        for b in range(self.wl.batch):
            gid, s = self.gids[b], self.orc.seqs[self.oids[b]]
            L = s.L
            if L == 0:
                continue
            pt = np.array(c.page_table(gid), np.int64)
            if Hd:
                assert len(pt) >= -(-L // P)
                t = np.arange(L)
                phys, row = pt[t // P], t % P
                nL = -(-L // ell)
                j = np.arange(nL)
                for hd, h in enumerate(self.dyn):
                    assert np.array_equal(kp[phys, hd, row], s.K[h, :L]), ("k_pool", b, h)
                    assert np.array_equal(vp[phys, hd, row], s.V[h, :L]), ("v_pool", b, h)
                    m = meta[pt[j // R], hd, j % R]
                    assert bits_equal(m[:, 0], s.kmin[h], mag), ("kmin", b, h)
                    assert bits_equal(m[:, 1], s.kmax[h], mag), ("kmax", b, h)
            for hs, h in enumerate(self.strm):
                T = oracle.streaming_tokens(L, S, Wn)
                slot = np.where(T < S, T, S + (T - S) % Wn)
                assert np.array_equal(sk[gid, hs, slot], s.K[h, T]), ("stream_k", b, h)
                assert np.array_equal(sv[gid, hs, slot], s.V[h, T]), ("stream_v", b, h)

    def check_selection(self, b, q):
        """GPU selection of every dynamic head of sequence b vs the oracle's."""
        gid, oid = self.gids[b], self.oids[b]
        s = self.orc.seqs[oid]
        info = self.cache.seq_info(gid)
        out = {}
        for h in self.dyn:
            g = np.array(self.cache.selection(gid, h), np.int32)
            o = s.sel[h]
            assert info["pages_at_selection"] == s.nL0[h]
            assert np.all(np.diff(g) > 0), "selection not strictly ascending"
            if not np.array_equal(g, o):
                S = self.orc.scores(oid, q, h)
                nL = s.nL0[h]
                assert len(g) == len(o) and g[-1] == nL - 1
                cand = np.setdiff1d(o, [nL - 1])
                cut = S[cand].min() if len(cand) else 0.0
                diff = np.setxor1d(g, o)
                tol = BAND * max(abs(float(cut)), 1e-30)
                assert np.all(np.abs(S[diff] - cut) <= tol), (
                    "selection differs beyond the tie band", b, h, diff, S[diff], cut)
            out[h] = g
        return out

    def step(self, step_idx, check_layout=False):
        """One decode step on both sides; returns (max_abs, mean_abs)."""
        wl, dt = self.wl, self.dt
        q, k, v = W.step_tokens(wl, step_idx, self.layer)
        out = self.cache.decode_step(tdev(q, dt, self.device), tdev(k, dt, self.device),
                                     tdev(v, dt, self.device), self.gids)
        self.cache.check_status()
        out = out.cpu().numpy().astype(np.float64)
        worst = (0.0, 0.0)
        for b in range(wl.batch):
            oid = self.oids[b]
            s = self.orc.seqs[oid]
            self.orc.append(oid, k[b][None], v[b][None])
            ran = self.orc.select(oid, q[b])
            gsel = self.check_selection(b, q[b]) if self.dyn else {}
            own = {h: s.sel[h] for h in self.dyn}
            same = all(np.array_equal(gsel[h], own[h]) for h in self.dyn)
            for h in self.dyn:
                s.sel[h] = gsel[h]
            ref = self.orc.attend(oid, q[b])
            for h in self.dyn:
                s.sel[h] = own[h]
            err = np.abs(out[b] - ref)
            mx, mean = float(err.max()), float(err.mean())
            assert np.isfinite(out[b]).all()
            assert mx <= TOL_MAX and mean <= TOL_MEAN, (step_idx, b, mx, mean)
            self.records.append(dict(step=step_idx, seq=b, selected=ran, same_sel=same,
                                     max_abs=mx, mean_abs=mean))
            worst = (max(worst[0], mx), max(worst[1], mean))
        if check_layout:
            self.check_layout()
        return worst
