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


def metric_of(workload):
    """The headline metric on its workload; the same quantity on the others."""
    if workload == "llama3_8b_b1_128k":
        return METRIC
    return "sparse decode attn us/step and KV GB/s (frac of ~8 TB/s HBM) on " + workload


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3_8b_b1_128k", choices=sorted(W.WORKLOADS))
    ap.add_argument("--layers", type=int, default=0,
                    help="layer instances (default: the workload's, at least 4x L2 touched "
                         "per step)")
    ap.add_argument("--replays", type=int, default=10,
                    help="timed replays of the K-step window (median, p10, p90 reported)")
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
    ap.add_argument("--no-dyn-only", action="store_true")
    ap.add_argument("--no-eager", action="store_true")
    ap.add_argument("--roofline-iters", type=int, default=40)
    ap.add_argument("--cpu-sample-steps", type=int, default=0,
                    help="oracle steps per CPU-baseline sample (default: the workload's)")
    return ap.parse_args()


# Layer instances per workload: enough that one step touches at least 4x the
# 129 MB L2 (KV bytes per layer-step x layers), so every step streams from HBM.
LAYERS = {"llama3_8b_b1_128k": 32, "llama3_8b_b4_32k": 16, "llama2_7b_mha_256k": 16,
          "cont_batch_16": 8, "tiny": 4}
# Oracle decode steps per CPU-baseline sample (about 10-30 s of host work at
# one thread on the slowest of them).
CPU_STEPS = {"llama3_8b_b1_128k": 8, "llama3_8b_b4_32k": 4, "llama2_7b_mha_256k": 2,
             "cont_batch_16": 2, "tiny": 8}
L2_BYTES = 129e6


def model_name(wl):
    return {(32, 8): "Llama-3-8B attention", (32, 32): "Llama-2-7B attention (MHA)"}.get(
        (wl.Hq, wl.Hkv), "synthetic attention")


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


def pct(xs):
    """(median, p10, p90) of a list."""
    a = np.asarray(xs, dtype=np.float64)
    return float(np.median(a)), float(np.percentile(a, 10)), float(np.percentile(a, 90))


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
    """n_layers independent caches of the workload, each holding the
    workload's batch of sequences at their context lengths."""

    FP8_SCALE = 1.0 / 32

    def __init__(self, wl, n_layers, device, extra_tokens, streaming_layers=(), kv_fp8=False):
        import torch
        import sparse_paged_decode_logical_gb300 as spd
        self.torch, self.wl, self.device = torch, wl, device
        lens = wl.seq_lens()
        self.lens = lens
        # per layer: the workload's head split, or every kv head streaming
        self.wls = [dataclasses.replace(wl, streaming=[True] * wl.Hkv)
                    if layer in streaming_layers else wl for layer in range(n_layers)]
        self.elem = 1 if kv_fp8 else 2
        self.caches, self.seqs = [], []
        for layer in range(n_layers):
            cfg = self.wls[layer].lib_config()
            cfg["max_context"] = max(lens) + extra_tokens
            cfg["num_physical_pages"] = sum(-(-(L + extra_tokens) // wl.P) for L in lens)
            if kv_fp8:
                cfg.update(kv_fp8=True, k_scale=[self.FP8_SCALE] * wl.Hkv,
                           v_scale=[self.FP8_SCALE] * wl.Hkv)
            c = spd.SparsePagedKVCache(device=device, **cfg)
            # every kernel on the stream is this library's and each layer's
            # cache is written only through its own context: the next layer
            # may stage its K/V tiles while the previous layer finishes
            c.set_early_kv_staging(True)
            ids = [c.seq_create() for _ in range(wl.batch)]
            for b, L in enumerate(lens):
                K, V = W.device_context(wl, b, L, layer, device)
                c.kv_append([ids[b]], K[None], V[None])
                del K, V
            self.caches.append(c)
            self.seqs.append(ids)
        torch.cuda.synchronize()
        tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
        self.tdt = tdt
        self.out = [torch.empty((wl.batch, wl.Hq, wl.d), dtype=torch.float32, device=device)
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
                k = torch.randn((wl.batch, wl.Hkv, wl.d), generator=self.gen,
                                device=self.device).to(self.tdt)
                v = torch.randn((wl.batch, wl.Hkv, wl.d), generator=self.gen,
                                device=self.device).to(self.tdt)
                row.append((q.contiguous(), k, v))
            res.append(row)
        return res

    def info(self):
        return self.caches[0].seq_info(self.seqs[0][0])

    def launches(self):
        return sum(c.launch_count() for c in self.caches)

    def layer_bytes(self, layer, selected):
        """(dyn, str, meta) bytes of the layer's current step, summed over its
        sequences (see step_bytes)."""
        tot = np.zeros(3)
        for sid in self.seqs[layer]:
            inf = self.caches[layer].seq_info(sid)
            n_att = (inf["pages_kept"] + (-(-inf["length"] // self.wl.ell))
                     - inf["pages_at_selection"])
            tot += step_bytes(self.wls[layer], inf["length"], n_att, selected, self.elem)
        return tot

    def step(self, row, outs=None):
        """Enqueue one decode step on every layer; returns its algorithmic bytes."""
        outs = outs or self.out
        due = self.info()["step_counter"] % self.wl.C == 0
        for layer, c in enumerate(self.caches):
            q, k, v = row[layer]
            c.decode_step(q, k, v, self.seqs[layer], out=outs[layer])
        tot = np.zeros(3)
        for layer in range(len(self.caches)):
            tot += self.layer_bytes(layer, due)
        return tot[0], tot[1], tot[2], due


def n_layers_of(args):
    return args.layers if args.layers > 0 else LAYERS.get(args.workload, 32)


def run_ours(args, rank, world, device):
    import torch
    torch.cuda.set_device(device)
    wl = W.workload(args.workload)
    n_l = n_layers_of(args)
    host_steps = 0 if args.no_eager else 4
    extra = args.warmup + args.steps + (0 if args.no_e2e else args.steps) + host_steps + 64
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

    # timed window: K steps captured into one graph.  The first replay runs
    # the K new steps; the window is then replayed again (each replay repeats
    # the same steps on the same inputs: appends rewrite the same slots, the
    # same pages are selected and attended, the same bytes are read) for the
    # spread over replays.
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
    reps = max(1, args.replays)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for r in range(reps):
            g.replay()
            evs[r + 1].record(stream)
    torch.cuda.synchronize()
    barrier()
    rep_ms = [max_over_ranks(evs[r].elapsed_time(evs[r + 1])) for r in range(reps)]
    ms, ms_p10, ms_p90 = pct(rep_ms)
    for c in layers.caches:
        c.check_status(stream)
    total_bytes = float(tot.sum())
    gbs = whole_job_gbs(total_bytes, ms, world)

    # roofline: the decode kernel alone (read-only, replayable), events around
    # every launch inside one graph; then the same for a context of the
    # workload's dynamic heads only (the selected-page bytes)
    rl = None if args.no_roofline else roofline(layers, stream, args.roofline_iters)
    if rl is not None:
        rl["exports"] = variant_timings(layers, stream)
        if not args.no_dyn_only and any(not s for s in wl.streaming) and \
                any(wl.streaming) and not streaming_layers(args):
            rl["dyn_only"] = dyn_only_roofline(wl, device, stream, args.roofline_iters,
                                               args.kv_fp8)
    clk = clocks.stop()

    # end to end: pinned host inputs -> device -> step -> pinned host outputs
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(layers, stream, args.steps, barrier, max_over_ranks, world)

    # eager launches (no graph): the host cost of the C-ABI decode step, and
    # the eager step time, for context
    host = None
    if not args.no_eager:
        host = host_cost(layers, stream, host_steps)

    peak, peak_kind = measured_peaks()
    res = {
        "metric": metric_of(args.workload),
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "us_per_step": ms / args.steps * 1e3,
        "us_per_layer_step": ms / args.steps / n_l * 1e3,
        "replays": {"n": reps, "ms_per_window_median": round(ms, 4),
                    "p10": round(ms_p10, 4), "p90": round(ms_p90, 4),
                    "first": round(rep_ms[0], 4),
                    "us_per_layer_step_p10_p90": [round(ms_p10 / args.steps / n_l * 1e3, 3),
                                                  round(ms_p90 / args.steps / n_l * 1e3, 3)]},
        "frac_of_hbm": round(gbs / world / peak, 4),
        "hbm_peak_gbs": peak,
        "hbm_peak_kind": peak_kind,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": data_desc(wl),
        "config": arm_config(wl, n_l, n_sel, total_bytes / args.steps, world,
                             streaming_layers(args), args.kv_fp8),
        "bytes_per_step": {"dyn": tot[0] / args.steps, "stream": tot[1] / args.steps,
                           "meta": tot[2] / args.steps},
        "gpu_launches": launches,
        "roofline": rl,
        "clocks": clk,
    }
    if host:
        res["host_us_per_layer_step"] = host["c_abi_us"]
        res["host"] = host
    if e2e:
        res["e2e"] = e2e
    return res, layers


def data_desc(wl):
    parts = ["seeded N(0,1) K/V in %s" % wl.dtype]
    if wl.outliers:
        parts.append("2 outlier key channels x50")
    if wl.needle == "pages":
        parts.append("needle pages at %s depth" % "/".join("%d%%" % (100 * f)
                                                           for f in wl.needle_depths))
    elif wl.needle == "tokens":
        parts.append("%.1f%% planted needle tokens" % (100 * wl.needle_frac))
    if wl.log_uniform_lens:
        parts.append("lengths log-uniform in [%dK, %dK]" % (wl.log_uniform_lens[0] // 1024,
                                                            wl.log_uniform_lens[1] // 1024))
    if wl.permute_pages:
        parts.append("physical pages in random order")
    return "synthetic (" + ", ".join(parts) + ")"


def streaming_layers(args):
    return sorted({int(x) for x in args.streaming_layers.split(",") if x.strip()})


def arm_config(wl, n_layers, n_sel=None, bytes_per_step=None, world=1, all_streaming=(),
               kv_fp8=False):
    lens = wl.seq_lens()
    c = {
        "workload": wl.name,
        "shape": "%s: %d q / %d kv heads, d %d, %s" % (model_name(wl), wl.Hq, wl.Hkv, wl.d,
                                                      wl.dtype),
        "context": wl.context if not wl.log_uniform_lens else
        "%d sequences, %d..%d tokens (sum %d)" % (len(lens), min(lens), max(lens), sum(lens)),
        "batch": wl.batch, "layers": n_layers,
        "logical_page": wl.ell, "physical_page": wl.P,
        "streaming_kv_heads": sum(wl.streaming), "sink": wl.sink, "window": wl.window,
        "token_budget": wl.token_budget if wl.token_budget > 0 else "min(4096, L/32)",
        "reuse_interval": wl.C,
        "l2": "inputs larger than L2: %d layers x %.0f MB touched per step" % (
            n_layers, (bytes_per_step or 0) / max(1, n_layers) / 1e6) if bytes_per_step else
        "inputs larger than L2",
        "timing": "timed window captured once into a CUDA graph and replayed (median over "
                  "replays); CUDA events on the launching stream; early KV staging on",
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
        "plain": lambda c, l: c.sparse_decode_attention(q[l], layers.seqs[l],
                                                        out=layers.out[l], stream=stream),
        "stats": lambda c, l: c.sparse_decode_attention_stats(q[l], layers.seqs[l],
                                                              stream=stream),
        "page_mass": lambda c, l: c.sparse_decode_attention_page_mass(
            q[l], layers.seqs[l], stream=stream),
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


def time_attention_graph(layers, stream, iters):
    """Median per-launch time (ms) of a graph of iters x n_layers back-to-back
    spd_sparse_decode_attention calls (one kernel each, the split combine is
    fused), replayed between CUDA events on the launching stream (read-only
    on the KV cache, so replays repeat identical work); at least 5 timed
    replays and about a second of them, so that the clock sampler sees the
    kernel under load.  Returns (ms per launch, launches per replay, replays,
    p10, p90)."""
    import torch
    n = len(layers.caches)
    row = layers.inputs(1)[0]
    q = [row[layer][0] for layer in range(n)]
    torch.cuda.synchronize()
    l0 = layers.launches()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(iters):
            for layer, c in enumerate(layers.caches):
                c.sparse_decode_attention(q[layer], layers.seqs[layer], out=layers.out[layer],
                                          stream=stream)
    per_replay = layers.launches() - l0
    times = []
    with torch.cuda.stream(stream):
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
    med, p10, p90 = pct(times)
    return med / per_replay, per_replay, len(times), p10 / per_replay, p90 / per_replay


def roofline(layers, stream, iters):
    """Average duration of the decode kernel (time_attention_graph) against
    the algorithmic bytes of one launch: the dynamic and streaming KV of one
    layer-step, averaged over the layers (they differ when some layers are
    all streaming)."""
    n = len(layers.caches)
    dyn = strm = 0.0
    for layer in range(n):
        d_, s_, _ = layers.layer_bytes(layer, False)
        dyn, strm = dyn + d_ / n, strm + s_ / n
    avg_ms, per_replay, n_rep, p10, p90 = time_attention_graph(layers, stream, iters)
    achieved = (dyn + strm) / (avg_ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    traffic = None
    tp = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    if os.path.exists(tp):
        # "key: value" lines written from an ncu capture of this kernel; the
        # figure is used only while the kernel sources are unchanged and the
        # workload is the one it was captured on
        kv = {}
        for ln in open(tp):
            if ":" in ln and not ln.startswith("#"):
                k, v = ln.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("kernel_source_hash") == kernel_hash() and layers.elem == 2 and \
                kv.get("workload", "llama3_8b_b1_128k") == layers.wl.name:
            try:
                traffic = float(kv["traffic_bytes_per_launch"])
            except (KeyError, ValueError):
                traffic = None
    return {"kernel": "decode_tiles_kernel (split-K sparse attention, fused combine), one layer",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": kind + " (MEASURED_PEAKS.json hbm_gbs, burst copy)" if kind == "measured" else kind,
            "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
            "algorithmic_bytes_per_launch": int(round(dyn + strm)),
            "avg_launch_us": round(avg_ms * 1e3, 3),
            "launch_us_p10_p90": [round(p10 * 1e3, 3), round(p90 * 1e3, 3)],
            "launches_per_replay": per_replay,
            "how": "graph of %d back-to-back decode launches (%d layers x %d), median over %d "
                   "replays / launches; includes inter-launch gaps" % (per_replay, n, iters, n_rep)}


def dyn_only_roofline(wl, device, stream, iters, kv_fp8=False, n_layers=48):
    """The decode kernel on the selected pages alone: contexts holding only
    the workload's dynamic kv heads (same shapes, budget and data
    distribution), n_layers of them (a round of launches reads more than 3x
    L2), timed like `roofline`; bytes per launch = the dynamic heads' |T| x d
    x 2 x element bytes."""
    import torch
    Hd = sum(1 for s in wl.streaming if not s)
    wd = dataclasses.replace(wl, Hkv=Hd, Hq=Hd * wl.G, streaming=[False] * Hd)
    lay = Layers(wd, n_layers, device, 64, kv_fp8=kv_fp8)
    with torch.cuda.stream(stream):
        for row in lay.inputs(2):
            lay.step(row)
    stream.synchronize()
    dyn = 0.0
    for layer in range(n_layers):
        dyn += lay.layer_bytes(layer, False)[0] / n_layers
    avg_ms, per_replay, n_rep, p10, p90 = time_attention_graph(lay, stream, iters)
    for c in lay.caches:
        c.check_status(stream)
    achieved = dyn / (avg_ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    del lay
    torch.cuda.empty_cache()
    return {"kernel": "decode_tiles_kernel on the dynamic heads only (selected pages)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "algorithmic_bytes_per_launch": int(round(dyn)),
            "avg_launch_us": round(avg_ms * 1e3, 3),
            "launch_us_p10_p90": [round(p10 * 1e3, 3), round(p90 * 1e3, 3)],
            "how": "%d contexts of %d dynamic kv heads (%d q heads), graph of %d back-to-back "
                   "launches, median over %d replays" % (n_layers, Hd, Hd * wl.G, per_replay,
                                                         n_rep)}


def host_cost(layers, stream, n_steps):
    """Host time of the decode step's C-ABI call, eager (no graph): every
    layer's spd_decode_step called through ctypes with pre-marshalled
    arguments for n_steps steps, timed on the host around the calls (the
    GPU keeps up: the device time per layer-step is shorter), then the
    same through the Python binding, and the eager step time with the GPU
    work included."""
    import ctypes
    import torch
    import sparse_paged_decode_logical_gb300 as spd
    L = spd.lib()
    n = len(layers.caches)
    rows = layers.inputs(2 * n_steps)
    st = ctypes.c_void_p(stream.cuda_stream)
    args = []
    for s_ in range(n_steps):
        row = []
        for layer, c in enumerate(layers.caches):
            q, k, v = rows[s_][layer]
            ids = (ctypes.c_int * len(layers.seqs[layer]))(*layers.seqs[layer])
            row.append((c.ctx, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                        ctypes.c_void_p(v.data_ptr()), ids, len(layers.seqs[layer]),
                        ctypes.c_void_p(layers.out[layer].data_ptr())))
        args.append(row)
    torch.cuda.synchronize()
    t_call = 0.0
    for row in args:
        for a in row:
            t0 = time.perf_counter()
            r = L.spd_decode_step(a[0], a[1], a[2], a[3], a[4], a[5], a[6], st)
            t_call += time.perf_counter() - t0
            assert r == 0
    stream.synchronize()
    # the Python binding (argument checks and marshalling included), and the
    # eager step time (host and GPU)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for s_ in range(n_steps, 2 * n_steps):
            for layer, c in enumerate(layers.caches):
                q, k, v = rows[s_][layer]
                c.decode_step(q, k, v, layers.seqs[layer], out=layers.out[layer])
    t_bind = time.perf_counter() - t0
    stream.synchronize()
    t_eager = time.perf_counter() - t0
    for c in layers.caches:
        c.check_status(stream)
    k = n_steps * n
    return {"c_abi_us": round(t_call / k * 1e6, 2),
            "binding_us": round(t_bind / k * 1e6, 2),
            "eager_us_per_layer_step": round(t_eager / k * 1e6, 2),
            "how": "host time of %d eager spd_decode_step calls (%d layers x %d steps) through "
                   "ctypes, then the same through the Python binding; eager = host enqueue "
                   "plus GPU, synchronized at the end" % (k, n, n_steps)}


# the sources the decode kernel is compiled from (its traffic figure is valid
# while they are unchanged)
DECODE_SOURCES = ("decode.cu", "decode_reuse.cu", "decode_kernel.cuh", "ptx.cuh", "spd_internal.h",
                  "topk.cuh")


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
    B = wl.batch
    rows = layers.inputs(n_steps)
    qn, kn = B * wl.Hq * wl.d, B * wl.Hkv * wl.d
    per_layer = qn + 2 * kn
    host_in = torch.empty((n_steps, n, per_layer), dtype=layers.tdt).pin_memory()
    for s_, row in enumerate(rows):
        for layer in range(n):
            q, k, v = row[layer]
            host_in[s_, layer] = torch.cat([q.reshape(-1), k.reshape(-1), v.reshape(-1)]).cpu()
    dev_in = torch.empty((n, per_layer), dtype=layers.tdt, device=layers.device)
    views = [(dev_in[layer, :qn].view(B, wl.Hq, wl.d),
              dev_in[layer, qn:qn + kn].view(B, wl.Hkv, wl.d),
              dev_in[layer, qn + kn:].view(B, wl.Hkv, wl.d)) for layer in range(n)]
    dev_out = torch.empty((n, B, wl.Hq, wl.d), dtype=torch.float32, device=layers.device)
    outs = [dev_out[layer] for layer in range(n)]
    host_out = torch.empty((n_steps, n, B, wl.Hq, wl.d), dtype=torch.float32).pin_memory()
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

def core_counts():
    """(threads available to this process (what nproc prints), online CPUs
    (the count std::thread::hardware_concurrency reports))."""
    avail = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    try:
        nproc = int(subprocess.run(["nproc"], capture_output=True, text=True).stdout.strip())
    except Exception:
        nproc = avail
    return nproc, os.cpu_count()


def oracle_sample(wl, n_steps, threads, warmup=0):
    """Time the oracle's decode steps (one layer, the workload's batch) on
    host cores, threads over kv heads.  Returns (GB/s, seconds per step,
    description)."""
    import oracle
    lens = wl.seq_lens()
    lay = oracle.OracleLayer(dict(
        num_q_heads=wl.Hq, num_kv_heads=wl.Hkv, head_dim=wl.d, dtype=wl.dtype,
        logical_page=wl.ell, streaming=wl.streaming, sink=wl.sink, window=wl.window,
        token_budget=wl.token_budget, reuse_interval=wl.C,
        max_context=max(lens) + warmup + n_steps + 8))
    sids = []
    for b, L in enumerate(lens):
        sid = lay.new_seq()
        K, V = W.context(wl, b, L)
        lay.append(sid, K, V)
        del K, V
        sids.append(sid)
    for s in range(warmup):
        q, k, v = W.step_tokens(wl, s)
        for b, sid in enumerate(sids):
            lay.step(sid, q[b], k[b], v[b], threads=threads)
    tot, t = 0.0, 0.0
    dh = [h for h in range(wl.Hkv) if not wl.streaming[h]]
    for s in range(warmup, warmup + n_steps):
        q, k, v = W.step_tokens(wl, s)
        dues = [lay.selection_due(sid) for sid in sids]
        t0 = time.perf_counter()
        for b, sid in enumerate(sids):
            lay.step(sid, q[b], k[b], v[b], threads=threads)
        t += time.perf_counter() - t0
        for b, sid in enumerate(sids):
            st = lay.seqs[sid]
            nL = -(-st.L // wl.ell)
            n_att = len(st.sel[dh[0]]) + nL - st.nL0[dh[0]] if dh else 0
            tot += sum(step_bytes(wl, st.L, n_att, dues[b]))
    desc = ("oracle decode steps (append + select when due + fp64 attention) of one layer "
            "of %s (%d sequence%s), %d steps, %d thread%s over kv heads"
            % (wl.name, len(lens), "s" if len(lens) > 1 else "", n_steps, threads,
               "s" if threads > 1 else ""))
    return tot / t / 1e9, t / n_steps, desc


def cpu_baseline(wl, n_steps):
    """The oracle at every available core and at one thread, same sample."""
    import oracle
    nproc, online = core_counts()
    threads = oracle.cpu_threads()
    gbs, sec, desc = oracle_sample(wl, n_steps, threads)
    gbs1, sec1, _ = oracle_sample(wl, n_steps, 1)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": desc, "ms_per_layer_step": round(sec * 1e3, 2),
            "value_1_thread": round(gbs1, 4), "ms_per_layer_step_1_thread": round(sec1 * 1e3, 2),
            "nproc": nproc, "hardware_concurrency": online}


def run_reference(args):
    import oracle
    wl = W.workload(args.workload)
    threads = oracle.cpu_threads()
    nproc, online = core_counts()
    gbs, sec, desc = oracle_sample(wl, args.steps, threads, args.warmup)
    return {
        "metric": metric_of(args.workload), "impl": "reference", "value": round(gbs, 4),
        "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": arm_config(wl, n_layers_of(args), all_streaming=streaming_layers(args)),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": desc, "nproc": nproc,
                         "hardware_concurrency": online},
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
    clocks = ClockSampler(device.index if device.index is not None else 0)
    clocks.start()
    times = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        out, blocks = spd.prefill_block_sparse_attention(q, k, v, wq, wk, blk, budget,
                                                         dense_below, check=False)
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    clk = clocks.stop()
    ms, ms_p10, ms_p90 = pct(times)
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
            "ms_p10_p90": [round(ms_p10, 3), round(ms_p90, 3)], "clocks": clk,
            "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tf / peak, 4) if peak else None,
                         "traffic": None,
                         "note": "attention FLOPs computed / time of the three kernels"}}


def main():
    args = parse()
    if args.prefill:
        import torch
        res = run_prefill(args.prefill, max(3, min(args.steps, 10)), max(1, min(args.warmup, 2)),
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
    res, layers = run_ours(args, rank, world, device)
    del layers
    torch.cuda.empty_cache()
    if rank == 0:
        if not args.no_cpu_baseline:
            wl = W.workload(args.workload)
            res["cpu_baseline"] = cpu_baseline(
                wl, args.cpu_sample_steps or CPU_STEPS.get(args.workload, 8))
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
