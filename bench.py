"""Benchmark: sparse decode attention at 128K context on GB300.

Workload (default): Llama-3-8B attention shapes -- 32 query / 8 kv heads,
head_dim 128, bf16 K/V -- one sequence at 131072 tokens, logical page 32,
physical page 1024, 4 streaming kv heads (sink 128 + window 4096) and 4
dynamic kv heads with budget min(4096, L/32) = 4096, selection reuse C = 4.
One "step" is one decode token through 32 independent layer instances of
that attention (the depth of Llama-3-8B): per layer, append the token and
update the page metadata, select pages when due, and run the split-K sparse
decode attention.  The 32 layers hold ~8.6 GB of K/V and touch ~610 MB per
step, so every step streams from HBM (inputs larger than the 129 MB L2).

Metric: KV GB/s = the bytes the sparse path must read (selected dynamic
pages + streaming sink/window + the metadata scanned on selection steps)
divided by the step time; also reported as microseconds per step and per
layer-step, with the fraction of the measured HBM bandwidth.

Arms:
  default            the CUDA library through its C ABI.  `value`: the timed
                     window of K steps (captured once into a CUDA graph, then
                     run once; inputs resident in HBM).  `e2e`: the same
                     metric with each step's q/k/v copied from pinned host
                     memory and the outputs copied back, inside the timed
                     region.  `roofline`: the decode kernel alone.
  --impl reference   the plain CPU oracle on the host cores, same metric,
                     on a bounded sample (one layer, the same seeded
                     128K workload).
"""
import argparse
import dataclasses
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "sparse decode attn us/step and KV GB/s (frac of ~8 TB/s HBM) at 128K context"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3_8b_b1_128k")
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--streaming-layers", default="",
                    help="comma-separated layer indices whose kv heads are all streaming "
                         "(the other layers keep the workload's head split)")
    ap.add_argument("--prefill", type=int, default=0, metavar="L",
                    help="time only the prefill block-sparse attention of one L-token prompt "
                         "(Llama-3-8B shapes, budget 4096, dense below 32K) and print its line")
    ap.add_argument("--kv-fp8", action="store_true",
                    help="store K/V as fp8 E4M3 codes (scale 1/32 on every kv head)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-roofline", action="store_true")
    ap.add_argument("--no-eager", action="store_true")
    ap.add_argument("--roofline-iters", type=int, default=40)
    ap.add_argument("--cpu-sample-steps", type=int, default=16)
    return ap.parse_args()


# ---- multi-rank aggregation (replicas: no data-path collective) -------------

def reduce_max(x, dist=None, device="cpu"):
    """Max of a host float over all ranks (identity on one process)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank, ms_max, world):
    """Weak scaling: every rank moves the same bytes; the job takes the
    slowest rank's time."""
    return bytes_per_rank * world / (ms_max * 1e-3) / 1e9


# ---- algorithmic bytes ------------------------------------------------------

def step_bytes(wl, L, n_att, selected, e=2):
    """Bytes one layer-step must read for one sequence of length L.

    n_att: attended logical pages per dynamic head (selection plus pages
    created since it).  Dynamic heads read every token of those pages (the
    last one holds L - (nL-1)*ell tokens); streaming heads read
    min(L, sink + window) tokens; a selection step also scans the min/max
    rows of the nL - 1 candidate pages.  e: bytes per stored element (2, or
    1 for fp8 storage)."""
    Hd = sum(1 for s in wl.streaming if not s)
    Hs = wl.Hkv - Hd
    nL = -(-L // wl.ell)
    last = L - (nL - 1) * wl.ell
    dyn_tok = (n_att - 1) * wl.ell + last if Hd else 0
    dyn = Hd * dyn_tok * wl.d * 2 * e
    strm = Hs * min(L, wl.sink + wl.window) * wl.d * 2 * e
    meta = 0
    if selected and Hd:
        K_sel = max(1, (wl.token_budget if wl.token_budget > 0 else min(4096, L // 32)) // wl.ell)
        if nL > K_sel:
            meta = Hd * (nL - 1) * 2 * wl.d * e
    return dyn, strm, meta


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---- clocks ------------------------------------------------------------------

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        # nvidia-smi numbers GPUs physically; address the one torch sees by UUID
        self.index = str(index)
        try:
            import torch
            u = str(torch.cuda.get_device_properties(index).uuid)
            self.index = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            if vis:
                self.index = vis.split(",")[index]
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), "spd_clocks_%d.csv" % os.getpid())

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.index, "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in open(self.path):
            t = [x.strip() for x in ln.split(",")]
            if len(t) < 9:
                continue
            try:
                sm.append(float(t[1]))
                mx.append(float(t[2]))
            except ValueError:
                continue
            for n, v in zip(names, t[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---- the CUDA arm ----------------------------------------------------------------

class Layers:
    """n_layers independent caches of the workload, one sequence each."""

    FP8_SCALE = 1.0 / 32

    def __init__(self, wl, n_layers, device, extra_tokens, streaming_layers=(), kv_fp8=False):
        import torch
        import sparse_paged_decode_logical_gb300 as spd
        self.torch, self.wl, self.device = torch, wl, device
        L0 = wl.context
        # per layer: the workload's head split, or every kv head streaming
        self.wls = [dataclasses.replace(wl, streaming=[True] * wl.Hkv)
                    if layer in streaming_layers else wl for layer in range(n_layers)]
        self.elem = 1 if kv_fp8 else 2
        self.caches, self.seqs = [], []
        for layer in range(n_layers):
            cfg = self.wls[layer].lib_config()
            cfg["max_context"] = L0 + extra_tokens
            cfg["max_seqs"] = 1
            cfg["num_physical_pages"] = -(-cfg["max_context"] // wl.P)
            if kv_fp8:
                cfg.update(kv_fp8=True, k_scale=[self.FP8_SCALE] * wl.Hkv,
                           v_scale=[self.FP8_SCALE] * wl.Hkv)
            c = spd.SparsePagedKVCache(device=device, **cfg)
            # every kernel on the stream is this library's and each layer's
            # cache is written only through its own context: the next layer
            # may stage its K/V tiles while the previous layer finishes
            c.set_early_kv_staging(True)
            s = c.seq_create()
            K, V = W.device_context(wl, 0, L0, layer, device)
            c.kv_append([s], K[None], V[None])
            del K, V
            self.caches.append(c)
            self.seqs.append(s)
        torch.cuda.synchronize()
        tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
        self.tdt = tdt
        self.out = [torch.empty((1, wl.Hq, wl.d), dtype=torch.float32, device=device)
                    for _ in range(n_layers)]
        self.u = [torch.from_numpy(W.query_base(wl, layer)).to(device) for layer in range(n_layers)]
        self.gen = torch.Generator(device=device)
        self.gen.manual_seed(20260 + wl.index)

    def inputs(self, n_steps):
        """Resident per-step inputs: list over steps of lists over layers of (q, k, v)."""
        torch, wl = self.torch, self.wl
        res = []
        for _ in range(n_steps):
            row = []
            for layer in range(len(self.caches)):
                q = (self.u[layer] + 0.25 * torch.randn(self.u[layer].shape, generator=self.gen,
                                                        device=self.device)).to(self.tdt)
                k = torch.randn((1, wl.Hkv, wl.d), generator=self.gen, device=self.device).to(self.tdt)
                v = torch.randn((1, wl.Hkv, wl.d), generator=self.gen, device=self.device).to(self.tdt)
                row.append((q.contiguous(), k, v))
            res.append(row)
        return res

    def info(self):
        return self.caches[0].seq_info(self.seqs[0])

    def launches(self):
        return sum(c.launch_count() for c in self.caches)

    def layer_bytes(self, layer, selected):
        """(dyn, str, meta) bytes of the layer's current step (see step_bytes)."""
        inf = self.caches[layer].seq_info(self.seqs[layer])
        n_att = inf["pages_kept"] + (-(-inf["length"] // self.wl.ell)) - inf["pages_at_selection"]
        return step_bytes(self.wls[layer], inf["length"], n_att, selected, self.elem)

    def step(self, row, outs=None):
        """Enqueue one decode step on every layer; returns its algorithmic bytes."""
        outs = outs or self.out
        due = self.info()["step_counter"] % self.wl.C == 0
        for layer, c in enumerate(self.caches):
            q, k, v = row[layer]
            c.decode_step(q, k, v, [self.seqs[layer]], out=outs[layer])
        tot = np.zeros(3)
        for layer in range(len(self.caches)):
            tot += self.layer_bytes(layer, due)
        return tot[0], tot[1], tot[2], due


def run_ours(args, rank, world, device):
    import torch
    torch.cuda.set_device(device)
    wl = W.workload(args.workload)
    n_l = args.layers
    extra = args.warmup + args.steps + (0 if args.no_e2e else args.steps) + 64
    layers = Layers(wl, n_l, device, extra, streaming_layers(args), args.kv_fp8)
    stream = torch.cuda.Stream(device=device)
    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()

    def max_over_ranks(x):
        return reduce_max(x, dist, device)

    # warm-up: W steps, enqueued on `stream`
    warm = layers.inputs(args.warmup)
    with torch.cuda.stream(stream):
        for row in warm:
            layers.step(row)
    stream.synchronize()
    for c in layers.caches:
        c.check_status(stream)

    # timed window: K steps captured into one graph, then run once
    rows = layers.inputs(args.steps)
    torch.cuda.synchronize()
    l0 = layers.launches()
    g = torch.cuda.CUDAGraph()
    tot = np.zeros(3)
    n_sel = 0
    with torch.cuda.graph(g, stream=stream):
        for row in rows:
            d_, s_, m_, due = layers.step(row)
            tot += (d_, s_, m_)
            n_sel += int(due)
    launches = layers.launches() - l0
    clocks = ClockSampler(device.index if device.index is not None else 0)
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t_start.record(stream)
        g.replay()
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(t_start.elapsed_time(t_end))
    for c in layers.caches:
        c.check_status(stream)
    total_bytes = float(tot.sum())
    gbs = whole_job_gbs(total_bytes, ms, world)

    # roofline: the decode kernel alone (read-only, replayable), events around
    # every launch inside one graph
    rl = None if args.no_roofline else roofline(layers, stream, args.roofline_iters)
    if rl is not None:
        rl["exports"] = variant_timings(layers, stream)
    clk = clocks.stop()

    # end to end: pinned host inputs -> device -> step -> pinned host outputs
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(layers, stream, args.steps, barrier, max_over_ranks, world)

    # eager launches (no graph), for context
    eager_us = float("nan")
    if not args.no_eager:
        eager_rows = layers.inputs(4)
        torch.cuda.synchronize()
        te0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for row in eager_rows:
                layers.step(row)
        stream.synchronize()
        eager_us = (time.perf_counter() - te0) / len(eager_rows) * 1e6

    peak, peak_kind = measured_peaks()
    res = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "us_per_step": ms / args.steps * 1e3,
        "us_per_layer_step": ms / args.steps / n_l * 1e3,
        "frac_of_hbm": round(gbs / world / peak, 4),
        "hbm_peak_gbs": peak,
        "hbm_peak_kind": peak_kind,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded N(0,1) K/V in bf16, needle pages at 10/50/90% depth)",
        "config": arm_config(wl, n_l, n_sel, total_bytes / args.steps, world,
                             streaming_layers(args), args.kv_fp8),
        "bytes_per_step": {"dyn": tot[0] / args.steps, "stream": tot[1] / args.steps,
                           "meta": tot[2] / args.steps},
        "gpu_launches": launches,
        "roofline": rl,
        "clocks": clk,
        "eager_us_per_step": round(eager_us, 1),
    }
    if e2e:
        res["e2e"] = e2e
    return res, layers


def streaming_layers(args):
    return sorted({int(x) for x in args.streaming_layers.split(",") if x.strip()})


def arm_config(wl, n_layers, n_sel=None, bytes_per_step=None, world=1, all_streaming=(),
               kv_fp8=False):
    c = {
        "workload": wl.name,
        "shape": "Llama-3-8B attention: 32 q / 8 kv heads, d 128, bf16",
        "context": wl.context, "batch": wl.batch, "layers": n_layers,
        "logical_page": wl.ell, "physical_page": wl.P,
        "streaming_kv_heads": sum(wl.streaming), "sink": wl.sink, "window": wl.window,
        "token_budget": "min(4096, L/32)", "reuse_interval": wl.C,
        "l2": "inputs larger than L2: %d layers x ~19 MB touched per step" % n_layers,
        "timing": "timed window captured once into a CUDA graph and run once; "
                  "CUDA events on the launching stream; early KV staging on",
        "parallelism": "replicas" if world > 1 else "single GPU",
    }
    if all_streaming:
        c["all_streaming_layers"] = list(all_streaming)
    if kv_fp8:
        c["kv_storage"] = "fp8 e4m3, scale %g per kv head" % Layers.FP8_SCALE
    if n_sel is not None:
        c["selection_steps_in_window"] = n_sel
    return c


def variant_timings(layers, stream, iters=10):
    """Per-launch time of the attention call with its optional exports, each
    timed like `roofline`: a graph of `iters` x n_layers back-to-back calls,
    median over replays.  plain: spd_sparse_decode_attention; stats: + row
    max / row sum; page_mass: + the dynamic heads' per-page attention mass."""
    import torch
    n = len(layers.caches)
    row = layers.inputs(1)[0]
    q = [row[layer][0] for layer in range(n)]
    calls = {
        "plain": lambda c, l: c.sparse_decode_attention(q[l], [layers.seqs[l]],
                                                        out=layers.out[l], stream=stream),
        "stats": lambda c, l: c.sparse_decode_attention_stats(q[l], [layers.seqs[l]],
                                                              stream=stream),
        "page_mass": lambda c, l: c.sparse_decode_attention_page_mass(
            q[l], [layers.seqs[l]], stream=stream),
    }
    res = {}
    for name, call in calls.items():
        torch.cuda.synchronize()
        l0 = layers.launches()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(iters):
                for layer, c in enumerate(layers.caches):
                    call(c, layer)
        per_replay = layers.launches() - l0
        times = []
        with torch.cuda.stream(stream):
            for rep in range(12):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g.replay()
                b.record(stream)
                b.synchronize()
                if rep:
                    times.append(a.elapsed_time(b))
        res[name + "_us_per_launch"] = round(float(np.median(times)) / per_replay * 1e3, 3)
    return res


def roofline(layers, stream, iters):
    """Average duration of the decode kernel: a graph of `iters` x n_layers
    back-to-back spd_sparse_decode_attention launches (one kernel each, the
    split combine is fused), replayed on the launching stream between CUDA
    events.  Read-only on the KV cache, so replays repeat identical work."""
    import torch
    wl = layers.wl
    n = len(layers.caches)
    row = layers.inputs(1)[0]
    q = [row[layer][0] for layer in range(n)]
    torch.cuda.synchronize()
    l0 = layers.launches()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(iters):
            for layer, c in enumerate(layers.caches):
                c.sparse_decode_attention(q[layer], [layers.seqs[layer]], out=layers.out[layer],
                                          stream=stream)
    per_replay = layers.launches() - l0
    # bytes per launch, averaged over the layers (they differ when some layers
    # are all streaming)
    dyn = strm = 0.0
    for layer in range(n):
        d_, s_, _ = layers.layer_bytes(layer, False)
        dyn, strm = dyn + d_ / n, strm + s_ / n
    times = []
    with torch.cuda.stream(stream):
        # at least 5 timed replays, and about a second of them so that the
        # clock sampler sees the kernel under load
        for rep in range(2000):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            if rep:
                times.append(a.elapsed_time(b))
            if len(times) >= 5 and sum(times) > 1000.0:
                break
    avg_ms = float(np.median(times)) / per_replay
    achieved = (dyn + strm) / (avg_ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    traffic = None
    tp = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    if os.path.exists(tp):
        # "key: value" lines written from an ncu capture of this kernel; the
        # figure is used only while the kernel sources are unchanged
        kv = {}
        for ln in open(tp):
            if ":" in ln and not ln.startswith("#"):
                k, v = ln.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("kernel_source_hash") == kernel_hash():
            try:
                traffic = float(kv["traffic_bytes_per_launch"])
            except (KeyError, ValueError):
                traffic = None
    return {"kernel": "decode_tiles_kernel (split-K sparse attention, fused combine), one layer",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": kind + " (MEASURED_PEAKS.json hbm_gbs, burst copy)" if kind == "measured" else kind,
            "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
            "algorithmic_bytes_per_launch": int(round(dyn + strm)),
            "avg_launch_us": round(avg_ms * 1e3, 3), "launches_per_replay": per_replay,
            "how": "graph of %d back-to-back decode launches (%d layers x %d), median over %d "
                   "replays / launches; includes inter-launch gaps" % (per_replay, n, iters,
                                                                        len(times))}


# the sources the decode kernel is compiled from (its traffic figure is valid
# while they are unchanged)
DECODE_SOURCES = ("decode.cu", "decode_kernel.cuh", "ptx.cuh", "spd_internal.h", "topk.cuh")


def kernel_hash():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_paged_decode_logical_gb300", "csrc")
    for f in DECODE_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def run_e2e(layers, stream, n_steps, barrier, max_over_ranks, world):
    """Per step: one H2D copy of every layer's q, k, v from pinned host memory
    into a device staging buffer, the decode step of every layer through the
    C ABI, and one D2H copy of every layer's output into pinned memory."""
    import torch
    wl = layers.wl
    n = len(layers.caches)
    rows = layers.inputs(n_steps)
    qn, kn = wl.Hq * wl.d, wl.Hkv * wl.d
    per_layer = qn + 2 * kn
    host_in = torch.empty((n_steps, n, per_layer), dtype=layers.tdt).pin_memory()
    for s_, row in enumerate(rows):
        for layer in range(n):
            q, k, v = row[layer]
            host_in[s_, layer] = torch.cat([q.reshape(-1), k.reshape(-1), v.reshape(-1)]).cpu()
    dev_in = torch.empty((n, per_layer), dtype=layers.tdt, device=layers.device)
    views = [(dev_in[layer, :qn].view(1, wl.Hq, wl.d), dev_in[layer, qn:qn + kn].view(1, wl.Hkv, wl.d),
              dev_in[layer, qn + kn:].view(1, wl.Hkv, wl.d)) for layer in range(n)]
    dev_out = torch.empty((n, 1, wl.Hq, wl.d), dtype=torch.float32, device=layers.device)
    outs = [dev_out[layer] for layer in range(n)]
    host_out = torch.empty((n_steps, n, 1, wl.Hq, wl.d), dtype=torch.float32).pin_memory()
    h2d = host_in[0].numel() * host_in.element_size()
    d2h = host_out[0].numel() * 4
    torch.cuda.synchronize()
    tot = 0.0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for s_ in range(n_steps):
            dev_in.copy_(host_in[s_], non_blocking=True)
            d_, st_, m_, _ = layers.step(views, outs=outs)
            tot += d_ + st_ + m_
            host_out[s_].copy_(dev_out, non_blocking=True)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(a.elapsed_time(b))
    assert bool(torch.isfinite(host_out[-1]).all())
    return {"value": round(whole_job_gbs(tot, ms, world), 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "us_per_step": round(ms / n_steps * 1e3, 2),
            "how": "per step: one H2D of every layer's q/k/v from pinned host memory, the "
                   "decode step of every layer through the C ABI, one D2H of every layer's "
                   "output; the window captured into one CUDA graph and run once"}


# ---- the CPU oracle arm ------------------------------------------------------------

def oracle_sample(wl, n_steps, warmup=0):
    """Time the oracle's decode steps (one layer, one sequence) on host cores.
    Returns (GB/s, seconds per step, threads, description)."""
    import oracle
    threads = oracle.cpu_threads()
    cfg = wl.lib_config()
    lay = oracle.OracleLayer(dict(
        num_q_heads=wl.Hq, num_kv_heads=wl.Hkv, head_dim=wl.d, dtype=wl.dtype,
        logical_page=wl.ell, streaming=wl.streaming, sink=wl.sink, window=wl.window,
        token_budget=wl.token_budget, reuse_interval=wl.C,
        max_context=wl.context + warmup + n_steps + 8))
    sid = lay.new_seq()
    K, V = W.context(wl, 0, wl.context)
    lay.append(sid, K, V)
    del K, V
    for s in range(warmup):
        q, k, v = W.step_tokens(wl, s)
        lay.step(sid, q[0], k[0], v[0], threads=threads)
    tot, t = 0.0, 0.0
    for s in range(warmup, warmup + n_steps):
        q, k, v = W.step_tokens(wl, s)
        due = lay.selection_due(sid)
        t0 = time.perf_counter()
        lay.step(sid, q[0], k[0], v[0], threads=threads)
        t += time.perf_counter() - t0
        st = lay.seqs[sid]
        dh = [h for h in range(wl.Hkv) if not wl.streaming[h]]
        nL = -(-st.L // wl.ell)
        n_att = len(st.sel[dh[0]]) + nL - st.nL0[dh[0]] if dh else 0
        tot += sum(step_bytes(wl, st.L, n_att, due))
    desc = ("oracle decode steps (append + select when due + fp64 attention) of one "
            "layer of %s at %d tokens, %d steps, threads over kv heads"
            % (wl.name, wl.context, n_steps))
    return tot / t / 1e9, t / n_steps, threads, desc


def run_reference(args):
    wl = W.workload(args.workload)
    gbs, sec, threads, desc = oracle_sample(wl, args.steps, args.warmup)
    return {
        "metric": METRIC, "impl": "reference", "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": arm_config(wl, args.layers, all_streaming=streaming_layers(args)),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_prefill(L, steps, warmup, device):
    """Prefill block-sparse attention of one L-token prompt with Llama-3-8B
    attention shapes (32 q / 8 kv heads, d 128, bf16, rank d/8): per step the
    three kernels (block means, selection, attention).  FLOP/s counts the
    attention actually computed: per query and head, 4 d flops for each key of
    its chosen blocks it may see (causal)."""
    import torch
    import sparse_paged_decode_logical_gb300 as spd
    Hq, Hkv, d, r, blk, budget, dense_below = 32, 8, 128, 16, 64, 4096, 32768
    g = torch.Generator(device=device)
    g.manual_seed(20262)
    q = torch.randn((L, Hq, d), generator=g, device=device).to(torch.bfloat16)
    k = torch.randn((L, Hkv, d), generator=g, device=device).to(torch.bfloat16)
    v = torch.randn((L, Hkv, d), generator=g, device=device).to(torch.bfloat16)
    wq = torch.randn((Hkv, d, r), generator=g, device=device) / d ** 0.5
    wk = torch.randn((Hkv, d, r), generator=g, device=device) / d ** 0.5
    for _ in range(warmup):
        spd.prefill_block_sparse_attention(q, k, v, wq, wk, blk, budget, dense_below, check=False)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        out, blocks = spd.prefill_block_sparse_attention(q, k, v, wq, wk, blk, budget,
                                                         dense_below, check=False)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    nb = -(-L // blk)
    keys = 0
    for bq in range(nb):
        n_sel = bq + 1 if L < dense_below else min(bq + 1, budget // blk)
        rows = min(blk, L - bq * blk)
        keys += (n_sel - 1) * blk * rows + rows * (rows + 1) // 2  # earlier blocks + causal own
    flops = keys * Hq * 4 * d
    peak = None
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        peak = json.load(open(pk)).get("bf16_tflops")
    tf = flops / (ms * 1e-3) / 1e12
    return {"metric": "prefill block-sparse attention ms per prompt", "value": round(ms, 3),
            "unit": "ms", "higher_is_better": False, "steps": steps, "warmup": warmup,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "prefill of one %d-token prompt, Llama-3-8B attention "
                                   "shapes, blocks of 64, budget 4096, rank 16" % L,
                       "dense": L < dense_below},
            "attention_tflops": round(tf, 2),
            "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tf / peak, 4) if peak else None,
                         "traffic": None,
                         "note": "attention FLOPs computed / time of the three kernels"}}


def main():
    args = parse()
    if args.prefill:
        import torch
        res = run_prefill(args.prefill, max(1, min(args.steps, 5)), max(1, min(args.warmup, 2)),
                          torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0"))))
        print(json.dumps(res), flush=True)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    res, _ = run_ours(args, rank, world, device)
    if rank == 0:
        if not args.no_cpu_baseline:
            wl = W.workload(args.workload)
            gbs, sec, threads, desc = oracle_sample(wl, args.cpu_sample_steps)
            res["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads,
                                   "kind": "oracle", "sample": desc,
                                   "ms_per_layer_step": round(sec * 1e3, 2)}
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
