#!/usr/bin/env python3
"""Benchmark of the attention path: prefill attention tokens/s and decode KV
GB/s against the GB300 roofline.

Workload (default): the attention-only 42-layer stack -- 5 sliding : 1 full
layers (sliding head_dim 256, window 512, theta 1e4; full head_dim 512, theta
1e6, partial rotary 0.25), n_heads 8, n_kv 2, the last 18 layers shared-KV --
at batch 8: prefill of T=4096 tokens, then 128 decode steps.  It is the one
workload that runs every step of the path (norm/RoPE/append, sliding and full
prefill attention, decode attention, shared-KV reads).  One benchmark step =
the whole job: prefill of all 42 layers, then the 128 decode steps (captured
in one CUDA graph).  Inputs are seeded N(0,1) bf16 drawn on the device; they
total ~10 GB per step, far above the 129 MB L2, so no L2 flush is needed.

value      prefill tokens/s: B*T / (prefill phase time).
decode     KV GB/s: algorithmic bytes of the 128 decode steps / decode phase time.
e2e        prefill tokens/s with the raw inputs copied host->device (pinned)
           and the last layer's output copied back, every step.
roofline   of the dominant kernel (most time per step), from CUDA events
           around its launches inside the timed steps.
configs    the other workloads (single-layer prefill, both decode workloads,
           the ring cache, the encoder form), each timed on its own with an
           L2 flush before every step and its own clock record.
cpu_baseline  the float64 oracle on all host cores, on a bounded sample.

  python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference]
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill attn tokens/s and decode KV GB/s vs GB300 roofline, 1 GPU"
WORKLOAD = "stack42_bf16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DECODE_EVENT_STEPS = (0, 32, 64, 96, 127)
# DRAM bytes (read + write) per launch from the ncu launch lists in
# profiles/ (dram__bytes_read.sum + dram__bytes_write.sum of each launch): the
# stack's kernels captured on the same stack at batch 2 (stack42_bf16_b2) and
# scaled by 4 to the benchmark's 8 sequences (every launch's bytes grow with
# the sequences it processes), the projections captured at the benchmark's
# own size.  Each figure carries the kernel's source files and the first 16
# hex digits of their SHA-256 at the capture: once the sources differ, the
# counters describe another kernel and the figure is not reported.
PREFILL_SOURCES = ("g4_prefill_tc.cu", "g4_device.cuh", "g4_internal.h")
DECODE_SOURCES = ("g4_attn_simt.cu", "g4_device.cuh", "g4_internal.h", "g4_normrope.cuh")
WIN_SOURCES = ("g4_decode_win.cu", "g4_device.cuh", "g4_internal.h", "g4_normrope.cuh")
GEMM_SOURCES = ("g4_gemm_tc.cu", "g4_device.cuh", "g4_internal.h", "g4_normrope.cuh")
PROFILED_TRAFFIC = {
    # key: (bytes per launch, sources, digest, where it comes from)
    "prefill_full": (521583616, PREFILL_SOURCES, "b1c7012b5f790912",
                     "ncu launch list, 42-layer stack at batch 2, layer-5 launches, x 4 sequences"),
    "decode_full": (134683648, DECODE_SOURCES, "9fdceb0610310b2d",
                    "ncu launch list, 42-layer stack at batch 2, full-layer decode steps, x 4 sequences"),
    "decode_sliding": (8710144, WIN_SOURCES, "b2ca64d9b97a6cb4",
                       "ncu launch list, 42-layer stack at batch 2, sliding-layer decode steps, x 4 sequences"),
    "qkv_sliding": (299278336, GEMM_SOURCES, "542a27ab55a5fddd", "ncu launch list, qkv_proj_bf16, sliding layer"),
    "qkv_full": (513194752, GEMM_SOURCES, "542a27ab55a5fddd", "ncu launch list, qkv_proj_bf16, full layer"),
    "out_sliding": (378548992, GEMM_SOURCES, "542a27ab55a5fddd", "ncu launch list, out_proj_bf16, sliding layer"),
    "out_full": (584822528, GEMM_SOURCES, "542a27ab55a5fddd", "ncu launch list, out_proj_bf16, full layer"),
}


def kernel_sources_hash(files):
    """First 16 hex digits of the SHA-256 of the concatenated kernel sources."""
    import hashlib
    m = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gemma_dual_geometry_gb300", "csrc", f), "rb") as fh:
            m.update(fh.read())
    return m.hexdigest()[:16]


def profiled_traffic(key):
    """(traffic per launch or None, where it comes from)."""
    if key not in PROFILED_TRAFFIC:
        return None, "no capture of this kernel"
    nbytes, files, digest, source = PROFILED_TRAFFIC[key]
    if kernel_sources_hash(files) != digest:
        return None, source + "; not reported: the kernel's sources changed after that capture"
    return nbytes, source


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload lines after the stack")
    ap.add_argument("--min-time", type=float, default=0.6,
                    help="seconds of timed steps each single-workload measurement runs at least (0: --steps only)")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--oracle-worker", default=None, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ---------------------------------------------------------------- multi-process plumbing

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def dist_init(backend):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x, device=None):
    """Maximum of a float over all ranks (identity on one process)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x, device=None):
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", str(self.gpu_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- workload arithmetic

def visible_pairs(T, window, sliding, q_start=0):
    """Sum over the T queries of the keys each one sees (causal, window)."""
    tot = 0
    for i in range(q_start, q_start + T):
        n = i + 1
        tot += min(n, window) if sliding else n
    return tot


def visible_pairs_bidirectional(T, window, sliding):
    """Sum over the T queries of the keys each one sees in the encoder form
    (|i - j| <= window on a sliding layer, all T otherwise)."""
    if not sliding:
        return T * T
    return sum(min(T, i + window + 1) - max(0, i - window) for i in range(T))


def prefill_flops(cfg, layer):
    from gemma_dual_geometry_gb300 import workloads as W
    g = W.layer_geometry(cfg, layer)
    if cfg.get("encoder"):
        pairs = visible_pairs_bidirectional(cfg["T"], g["window"], g["layer_type"] == W.SLIDING)
    else:
        pairs = visible_pairs(cfg["T"], g["window"], g["layer_type"] == W.SLIDING)
    return 4.0 * g["head_dim"] * cfg["H"] * cfg["B"] * pairs  # QK^T and PV, 2 flops per MAC


def decode_bytes(cfg, layer, L):
    """Algorithmic HBM bytes of one decode attention call at length L: the
    visible K and V rows, the q read and the output write."""
    from gemma_dual_geometry_gb300 import workloads as W
    g = W.layer_geometry(cfg, layer)
    keys = min(L, g["window"]) if g["layer_type"] == W.SLIDING else L
    hd, B = g["head_dim"], cfg["B"]
    return B * (keys * cfg["Hkv"] * hd * 2 * 2 + 2 * cfg["H"] * hd * 2)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- the GPU arm

class Job:
    """Device buffers and launch sequences of one benchmark step."""

    def __init__(self, cfg, device):
        import torch

        from gemma_dual_geometry_gb300 import workloads as W
        from gemma_dual_geometry_gb300.stack import AttnStack

        self.cfg, self.W, self.torch = cfg, W, torch
        self.B, self.T, self.S = cfg["B"], cfg["T"], cfg["decode_steps"]
        self.Lmax = self.T + self.S
        self.st = AttnStack(cfg, self.Lmax, device=device)
        self.n = self.st.n
        dev = device
        H, Hkv, dt = cfg["H"], cfg["Hkv"], cfg["dtype"]
        tdt = W.torch_dtype(dt)
        hds = sorted({g["head_dim"] for g in self.st.geo})
        # prefill inputs (raw projections) and decode inputs, per layer
        self.X, self.D = [], []
        for l in range(self.n):
            owns = self.st.owns(l)
            x = W.layer_inputs(cfg, l, self.T, owns, device=dev)
            x["q_norm_w"] = x["q_norm_w"].to(dev)
            if owns:
                x["k_norm_w"] = x["k_norm_w"].to(dev)
            self.X.append(x)
            hd = self.st.geo[l]["head_dim"]
            s = cfg["seed"]
            d = dict(q=W.normal((self.S, self.B, 1, H, hd), W.seed_for(s, l, 7), dt, dev))
            if owns:
                d["k"] = W.normal((self.S, self.B, 1, Hkv, hd), W.seed_for(s, l, 8), dt, dev)
                d["v"] = W.normal((self.S, self.B, 1, Hkv, hd), W.seed_for(s, l, 9), dt, dev)
            self.D.append(d)
        self.pos_pf = torch.arange(self.T, dtype=torch.int32, device=dev).repeat(self.B, 1).contiguous()
        self.qs = torch.zeros(self.B, dtype=torch.int32, device=dev)
        self.pos_dec = (self.T + torch.arange(self.S, dtype=torch.int32, device=dev))[:, None].repeat(1, self.B)
        self.pos_dec = self.pos_dec.contiguous()
        self.sl_dec = (self.pos_dec + 1).contiguous()
        self.qo = {hd: torch.empty((self.B, self.T, H, hd), dtype=tdt, device=dev) for hd in hds}
        self.out = {hd: torch.empty((self.B, self.T, H, hd), dtype=tdt, device=dev) for hd in hds}
        self.qo_dec = {hd: torch.empty((self.B, 1, H, hd), dtype=tdt, device=dev) for hd in hds}
        self.out_dec = {hd: torch.empty((self.B, H, hd), dtype=tdt, device=dev) for hd in hds}
        self.full_layers = [l for l in range(self.n) if self.st.geo[l]["layer_type"] == W.FULL]
        self.sliding_layers = [l for l in range(self.n) if self.st.geo[l]["layer_type"] == W.SLIDING]
        # decode launches timed with events, as spans (first layer, count):
        # every full layer alone, and the first run of consecutive sliding
        # layers that own their cache and the first that share one.  A span
        # runs from the end of the launch before it to the end of its last
        # launch (the events are graph leaves, see decode())
        def first_run(ls):
            run = ls[:1]
            while run and run[-1] + 1 in ls:
                run.append(run[-1] + 1)
            return [(run[0], len(run))] if run else []
        own = [l for l in self.sliding_layers if self.st.owns(l)]
        shared = [l for l in self.sliding_layers if not self.st.owns(l)]
        self.dec_timed_spans = [(l, 1) for l in self.full_layers] + first_run(own) + first_run(shared)
        self.pf_events = []
        self.dec_events = []
        self.graph = None

    # one pass of prefill over all layers
    def prefill(self, record=False):
        torch = self.torch
        for l in range(self.n):
            x, hd = self.X[l], self.st.geo[l]["head_dim"]
            self.st.append(l, x["q"], x.get("k"), x.get("v"), x["q_norm_w"], x.get("k_norm_w"), self.pos_pf,
                           self.T, self.qo[hd])
            ev = None
            if record and l in self.full_layers:
                ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                ev[0].record()
            self.st.prefill_attn(l, self.qo[hd], self.qs, self.T, self.out[hd])
            if ev is not None:
                ev[1].record()
                self.pf_events.append(ev)

    def decode(self, events=None, side=None):
        """One pass of decode steps.  With events (inside a graph capture), a
        span's start and end events are recorded on the side stream, each
        after the launch before it: a leaf of the graph that no launch waits
        for, so the chain of launches and their programmatic-dependent-launch
        overlap stay as they are without events."""
        torch = self.torch
        H, Hkv = self.cfg["H"], self.cfg["Hkv"]
        ends = {}
        if events:
            for (s, l0), (e0, e1, n) in events.items():
                ends[(s, l0 + n - 1)] = e1

        def mark(e):
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                e.record()

        for s in range(self.S):
            for l in range(self.n):
                d, hd = self.D[l], self.st.geo[l]["head_dim"]
                ev = events.get((s, l)) if events else None
                if ev is not None:
                    mark(ev[0])
                ev = ends.get((s, l))
                self.st.decode_step(l, d["q"][s].view(self.B, H, hd),
                                    d["k"][s].view(self.B, Hkv, hd) if "k" in d else None,
                                    d["v"][s].view(self.B, Hkv, hd) if "v" in d else None,
                                    self.X[l]["q_norm_w"], self.X[l].get("k_norm_w"), self.sl_dec[s], self.Lmax,
                                    self.out_dec[hd])
                if ev is not None:
                    mark(ev)
        if events:
            torch.cuda.current_stream().wait_stream(side)

    def capture_decode(self):
        torch = self.torch
        events = {}
        try:
            for s in sorted({s for s in DECODE_EVENT_STEPS if s < self.S} | {self.S - 1}):
                for l, n in self.dec_timed_spans:
                    events[(s, l)] = (torch.cuda.Event(enable_timing=True, external=True),
                                      torch.cuda.Event(enable_timing=True, external=True), n)
        except TypeError:
            events = {}
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.decode()  # warm-up outside capture (attributes, symbol addresses)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        mark_stream = torch.cuda.Stream()
        with torch.cuda.graph(self.graph):
            self.decode(events, side=mark_stream)
        torch.cuda.synchronize()
        self.dec_events = list(events.items())

    def launches_per_step(self):
        pf = 2 * self.n
        dec = self.S * sum(self.st.decode_launches(l) for l in range(self.n))
        return pf + dec

    def decode_step_bytes(self):
        return sum(decode_bytes(self.cfg, l, self.T + s + 1) for s in range(self.S) for l in range(self.n))


def run_ours(args, cfg):
    import torch

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dist_init("nccl")
    dev = torch.device("cuda", local)
    from gemma_dual_geometry_gb300 import build as g4build
    from gemma_dual_geometry_gb300 import g4attn as G
    g4build.build()
    G.lib()

    job = Job(cfg, dev)
    job.capture_decode()
    B, T = cfg["B"], cfg["T"]

    # warm-up
    for _ in range(args.warmup):
        job.prefill()
        job.graph.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(_gpu_uuid(dev))
    ev_pf = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
              torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    job.pf_events = []
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_wall0 = time.perf_counter()
    ev_all0 = torch.cuda.Event(enable_timing=True)
    ev_all1 = torch.cuda.Event(enable_timing=True)
    ev_all0.record()
    dec_samples = []
    for i in range(args.steps):
        ev_pf[i][0].record()
        job.prefill(record=True)
        ev_pf[i][1].record()
        job.graph.replay()
        ev_pf[i][2].record()
        if job.dec_events and i == args.steps - 1:
            pass
    ev_all1.record()
    torch.cuda.synchronize()
    barrier()
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    # decode kernel events hold the last replay's timings
    for (s, l), (e0, e1, n) in job.dec_events:
        dec_samples.append((s, l, e0.elapsed_time(e1) * 1e-3 / n, n))  # time per launch, launches

    total_s = ev_all0.elapsed_time(ev_all1) * 1e-3
    pf_s = sum(e[0].elapsed_time(e[1]) for e in ev_pf) * 1e-3
    dec_s = sum(e[1].elapsed_time(e[2]) for e in ev_pf) * 1e-3
    total_s = reduce_max(total_s, dev)
    pf_s = reduce_max(pf_s, dev)
    dec_s = reduce_max(dec_s, dev)

    tokens = B * T * args.steps * world
    value = tokens / pf_s
    dec_bytes = job.decode_step_bytes()
    dec_gbs = dec_bytes * args.steps * world / dec_s / 1e9

    peaks, peak_src = load_peaks()
    # prefill dominant kernel: tcgen05 attention of the full layers
    pf_launch = [e[0].elapsed_time(e[1]) * 1e-3 for e in job.pf_events]
    fl = job.full_layers[0]
    pf_flops = prefill_flops(cfg, fl)
    pf_avg = statistics.mean(pf_launch)
    rl_prefill = dict(kernel="prefill_tc_kernel<512> (full layer, tcgen05)", bound="tensor",
                      achieved=pf_flops / pf_avg / 1e12, peak=peaks["bf16_tflops_sustained"], unit="TFLOP/s",
                      peak_kind=f"{peak_src} bf16 dense, sustained (timed inside a long step)",
                      flops_per_launch=pf_flops, avg_launch_ms=pf_avg * 1e3, launches_sampled=len(pf_launch),
                      launches_per_step=len(job.full_layers))
    rl_prefill["traffic"], rl_prefill["traffic_source"] = profiled_traffic("prefill_full")
    rl_prefill["frac"] = rl_prefill["achieved"] / rl_prefill["peak"]
    rl_prefill["frac_of_burst"] = rl_prefill["achieved"] / peaks["bf16_tflops"]
    rooflines = [rl_prefill]
    kinds = (("full", job.full_layers, "attn_simt_kernel<bf16,512,4,fused> (full-layer decode step: append + "
                                       "split-KV attention + last-CTA merge)"),
             ("sliding", job.sliding_layers, "decode_win_kernel<256,4,fused> (sliding-layer decode step, window "
                                             "512: append + a cluster of eight 64-key CTAs merged in the leader's "
                                             "shared memory)"))
    for kind, layers, name in kinds:
        samples = [(s, l, t) for (s, l, t, _) in dec_samples if l in layers]
        n_launches = sum(n for (_, l, _, n) in dec_samples if l in layers)
        if not samples:
            continue
        per = [decode_bytes(cfg, l, T + s + 1) / t for (s, l, t) in samples]
        avg_t = statistics.mean(t for (_, _, t) in samples)
        avg_b = statistics.mean(decode_bytes(cfg, l, T + s + 1) for (s, l, _) in samples)
        rl_dec = dict(kernel=name, bound="hbm",
                      achieved=avg_b / avg_t / 1e9, peak=peaks["hbm_gbs"], unit="GB/s",
                      peak_kind=f"{peak_src} HBM copy bandwidth", bytes_per_launch=avg_b,
                      avg_launch_ms=avg_t * 1e3, launches_sampled=n_launches,
                      launches_per_step=len(layers) * cfg["decode_steps"],
                      per_launch_gbs_min=min(per) / 1e9, per_launch_gbs_max=max(per) / 1e9)
        rl_dec["traffic"], rl_dec["traffic_source"] = profiled_traffic("decode_" + kind)
        rl_dec["frac"] = rl_dec["achieved"] / rl_dec["peak"]
        if kind == "sliding":
            rl_dec["note"] = ("latency-bound: %.1f MB per launch, so the kernel's chain of dependent phases "
                              "(cos/sin table, norm, scores, softmax, P.V, cluster merge) outweighs the "
                              "streaming; timed over runs of 5 consecutive sliding layers, from the end of the "
                              "launch before the run to the end of its last launch (events recorded off the "
                              "chain of launches)" % (avg_b / 1e6))
        rooflines.append(rl_dec)
    # the dominant kernel is the one with the most time per step
    dominant = max(rooflines, key=lambda r: r["avg_launch_ms"] * r["launches_per_step"])

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_s / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), on device)",
        "config": {"workload": f"{args.workload}: attention-only 42-layer stack (5 sliding : 1 full, last 18 "
                               f"shared-KV), n_heads 8, n_kv 2, head_dim 256 / global 512, window 512, batch {B} "
                               f"per GPU, prefill T={T} then {cfg['decode_steps']} decode steps",
                   "global_batch": B * world, "seq_len": T, "decode_steps": cfg["decode_steps"],
                   "parallelism": f"replicas x{world} (independent sequences, no collective)",
                   "l2": "inputs larger than L2 (~10 GB per step), no flush",
                   "value_definition": "B*T prefill tokens / prefill-phase time (CUDA events)"},
        "ms_prefill_per_step": pf_s / args.steps * 1e3, "ms_decode_per_step": dec_s / args.steps * 1e3,
        "decode": {"value": dec_gbs, "unit": "GB/s", "frac_of_hbm": dec_gbs / peaks["hbm_gbs"],
                   "bytes_per_step": dec_bytes, "note": f"algorithmic KV + q + out bytes of {cfg['decode_steps']} steps x 42 "
                                                         f"layers / decode-phase time (one CUDA graph of fused "
                                                         f"decode steps)"},
        "roofline": dominant, "rooflines": rooflines,
        "gpu_launches": job.launches_per_step() * args.steps, "clocks": clk,
        "wall_s_timed_region": t_wall,
    }

    if not args.no_e2e:
        line["e2e"] = run_e2e(job, args, dev, world)
    del job
    torch.cuda.empty_cache()
    if not args.no_configs:
        # the other workloads, each measured on its own (own L2 flush, own clocks)
        line["configs"] = {name: measure_layer_workload(name, args, dev) for name in EXTRA_WORKLOADS}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, steps=1, warmup=0)
    if rank == 0:
        print(json.dumps(line), flush=True)


class LayerJob:
    """One- or two-layer workloads: single-layer prefill (prefill_bf16), the
    encoder form (encoder_bf16), or decode against prefilled caches
    (decode_bf16, ring_decode_bf16, longctx_decode_bf16).  A step is append +
    attention for every layer of the workload."""

    def __init__(self, cfg, device):
        import torch

        from gemma_dual_geometry_gb300 import workloads as W
        from gemma_dual_geometry_gb300.stack import AttnStack

        self.cfg, self.W, self.torch = cfg, W, torch
        self.B = cfg["B"]
        self.decode = "T" not in cfg
        self.encoder = bool(cfg.get("encoder"))
        H, Hkv, dt = cfg["H"], cfg["Hkv"], cfg["dtype"]
        if self.decode:
            if "L" in cfg:
                self.L = [cfg["L"]] * self.B
            else:
                self.L = [int(x) for x in W.lengths(self.B, cfg["L_lo"], cfg["L_hi"], cfg["seed"])]
            self.Lmax = max(self.L)
            self.T = 1
        else:
            self.T = cfg["T"]
            self.Lmax = self.T
        self.st = AttnStack(cfg, self.Lmax, device=device)
        self.n = self.st.n
        if self.decode:
            for l in range(self.n):
                k, v = W.prefilled_cache(cfg, l, W.cache_rows(cfg, l, self.Lmax), device=device)
                self.st.caches[l][0].copy_(k)
                self.st.caches[l][1].copy_(v)
                del k, v
        self.X = []
        for l in range(self.n):
            x = W.layer_inputs(cfg, l, self.T, True, device=device)
            x["q_norm_w"] = x["q_norm_w"].to(device)
            x["k_norm_w"] = x["k_norm_w"].to(device)
            self.X.append(x)
        if self.decode:
            self.pos = torch.tensor([[L - 1] for L in self.L], dtype=torch.int32, device=device)
            self.sl = torch.tensor(self.L, dtype=torch.int32, device=device)
        else:
            self.pos = torch.arange(self.T, dtype=torch.int32, device=device).repeat(self.B, 1).contiguous()
            self.qs = torch.zeros(self.B, dtype=torch.int32, device=device)
        self.qo = [torch.empty_like(x["q"]) for x in self.X]
        self.out = [torch.empty_like(x["q"]) for x in self.X]
        self.events = {l: [] for l in range(self.n)}

    def step(self, record=False):
        torch = self.torch
        H, Hkv = self.cfg["H"], self.cfg["Hkv"]
        for l in range(self.n):
            x, hd = self.X[l], self.st.geo[l]["head_dim"]
            if not self.decode:
                self.st.append(l, x["q"], x["k"], x["v"], x["q_norm_w"], x["k_norm_w"], self.pos, self.T,
                               self.qo[l])
            ev = None
            if record:
                ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                ev[0].record()
            if self.decode:
                self.st.decode_step(l, x["q"].view(self.B, H, hd), x["k"].view(self.B, Hkv, hd),
                                    x["v"].view(self.B, Hkv, hd), x["q_norm_w"], x["k_norm_w"], self.sl, self.Lmax,
                                    self.out[l].view(self.B, H, hd))
            elif self.encoder:
                self.st.encoder_attn(l, self.qo[l], self.T, self.out[l])
            else:
                self.st.prefill_attn(l, self.qo[l], self.qs, self.T, self.out[l])
            if ev is not None:
                ev[1].record()
                self.events[l].append(ev)

    def layer_work(self, l):
        """Algorithmic flops (prefill) or bytes (decode) of one attention launch of layer l."""
        if self.decode:
            return sum(decode_bytes(dict(self.cfg, B=1), l, L) for L in self.L)
        return prefill_flops(self.cfg, l)

    def launches_per_step(self):
        if self.decode:
            return sum(self.st.decode_launches(l) for l in range(self.n))
        return 2 * self.n


class ProjJob:
    """The projection workloads (qkv_proj_bf16, out_proj_bf16): one step is
    the fused projection of every layer of the workload, each launch timed
    with CUDA events like LayerJob's attention launches."""

    decode = False
    encoder = False

    def __init__(self, cfg, device):
        import torch

        from gemma_dual_geometry_gb300 import g4attn as G
        from gemma_dual_geometry_gb300 import workloads as W
        from gemma_dual_geometry_gb300.stack import AttnStack

        self.cfg, self.torch, self.G = cfg, torch, G
        self.B, self.T, self.D = cfg["B"], cfg["T"], cfg["D"]
        self.M = self.B * self.T
        self.kind = cfg["proj"]
        self.st = AttnStack(cfg, self.T, device=device) if self.kind == "qkv" else None
        self.geo = [W.layer_geometry(cfg, l) for l in range(len(cfg["types"]))]
        self.n = len(self.geo)
        self.X = [W.projection_inputs(cfg, l, device=device) for l in range(self.n)]
        if self.kind == "qkv":
            self.pos = torch.arange(self.T, dtype=torch.int32, device=device).repeat(self.B, 1).contiguous()
            self.qo = [torch.empty((self.M, cfg["H"], g["head_dim"]), dtype=torch.bfloat16, device=device)
                       for g in self.geo]
        else:
            self.out = [torch.empty((self.M, self.D), dtype=torch.bfloat16, device=device) for _ in self.geo]
        self.events = {l: [] for l in range(self.n)}

    def step(self, record=False):
        torch, G = self.torch, self.G
        for l in range(self.n):
            x = self.X[l]
            ev = None
            if record:
                ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                ev[0].record()
            if self.kind == "qkv":
                G.g4_qkv_project_append(self.st.params[l], self.st.table, l, x["x"], self.D, x["w"], x["q_norm_w"],
                                        x["k_norm_w"], self.pos, self.B, self.T, self.qo[l])
            else:
                K = self.cfg["H"] * self.geo[l]["head_dim"]
                G.g4_attn_out_residual(x["ao"], self.M, K, x["w"], self.D, x["post_w"], self.geo[l]["eps"], x["h"],
                                       self.out[l])
            if ev is not None:
                ev[1].record()
                self.events[l].append(ev)

    def layer_work(self, l):
        """Algorithmic flops of one launch: 2 M N K of the GEMM."""
        hd, H, Hkv = self.geo[l]["head_dim"], self.cfg["H"], self.cfg["Hkv"]
        if self.kind == "qkv":
            return 2.0 * self.M * (H + 2 * Hkv) * hd * self.D
        return 2.0 * self.M * self.D * H * hd

    def label(self, l):
        g = self.geo[l]
        if self.kind == "qkv":
            return (f"gemm_tc_kernel<{g['head_dim']},0>: q/k/v projection (M {self.M}, N "
                    f"{(self.cfg['H'] + 2 * self.cfg['Hkv']) * g['head_dim']}, K {self.D}) + input norm + per-head "
                    f"norm / RoPE / append")
        return (f"gemm_tc_kernel<256,1>: o_proj (M {self.M}, N {self.D}, K {self.cfg['H'] * g['head_dim']}) + "
                f"post-attention norm + residual")

    def launches_per_step(self):
        return self.n


L2_FLUSH_BYTES = 256 << 20   # written before every step of the per-workload measurements (> the 129 MB L2)
# The workloads measured after the stack in the default run (one entry each
# under "configs" of the JSON line, each with its own clock record).
EXTRA_WORKLOADS = ("prefill_bf16", "decode_bf16", "longctx_decode_bf16", "ring_decode_bf16", "encoder_bf16",
                   "qkv_proj_bf16", "out_proj_bf16")


def measure_layer_workload(name, args, dev, min_timed_s=None, max_steps=4000):
    """Times one of the one- or two-layer workloads on its own.

    Every step (append + attention of each layer, or the fused decode step) is
    preceded by a 256 MB write that flushes the L2, outside the step's CUDA
    events; the step count grows until the timed steps add up to at least
    ``min_timed_s`` so the nvidia-smi clock record (sampled every 200 ms
    while they run) has samples.  Returns a dict: the workload's value
    (prefill tokens/s or decode KV GB/s), per-layer rooflines from CUDA events
    around each attention launch, and the clocks."""
    import torch
    from gemma_dual_geometry_gb300 import workloads as W
    if min_timed_s is None:
        min_timed_s = args.min_time
    cfg = W.CONFIGS[name]
    job = ProjJob(cfg, dev) if cfg.get("proj") else LayerJob(cfg, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        job.step()
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record()
    job.step()
    c1.record()
    torch.cuda.synchronize()
    per_step = max(c0.elapsed_time(c1) * 1e-3, 1e-6)
    steps = int(min(max_steps, max(args.steps, -(-min_timed_s // per_step) if min_timed_s > 0 else 0)))
    job.events = {l: [] for l in range(job.n)}
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    clocks = ClockSampler(_gpu_uuid(dev))
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    for i in range(steps):
        flush.zero_()
        ev[i][0].record()
        job.step(record=True)
        ev[i][1].record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    total = reduce_max(sum(a.elapsed_time(b) for a, b in ev) * 1e-3, dev)
    _, world, _ = dist_env()
    peaks, src = load_peaks()
    per_layer = []
    for l in range(job.n):
        t = statistics.mean(a.elapsed_time(b) for a, b in job.events[l]) * 1e-3
        w = job.layer_work(l)
        g = job.geo[l] if isinstance(job, ProjJob) else job.st.geo[l]
        r = dict(layer=l, layer_type="sliding" if g["layer_type"] == 0 else "full", head_dim=g["head_dim"],
                 avg_launch_ms=t * 1e3, launches_sampled=len(job.events[l]), traffic=None)
        if job.decode:
            ach = w / t / 1e9
            r.update(kernel="decode step (append of the new token + split-KV attention + merge)", bound="hbm",
                     achieved=ach, peak=peaks["hbm_gbs"], unit="GB/s", frac=ach / peaks["hbm_gbs"],
                     bytes_per_launch=w, peak_kind=f"{src} HBM copy bandwidth")
        else:
            ach = w / t / 1e12
            r.update(kernel=job.label(l) if isinstance(job, ProjJob) else
                     "tcgen05 " + ("encoder" if job.encoder else "prefill") + " attention", bound="tensor",
                     achieved=ach, peak=peaks["bf16_tflops"], unit="TFLOP/s", frac=ach / peaks["bf16_tflops"],
                     frac_of_sustained=ach / peaks["bf16_tflops_sustained"], flops_per_launch=w,
                     peak_kind=f"{src} bf16 dense, burst (kernel timed alone; frac_of_sustained against the "
                               f"sustained peak)")
        if isinstance(job, ProjJob):
            r["traffic"], r["traffic_source"] = profiled_traffic(f"{job.kind}_{r['layer_type']}")
        per_layer.append(r)
    if job.decode:
        step_bytes = sum(job.layer_work(l) for l in range(job.n))
        value, unit = step_bytes * steps * world / total / 1e9, "GB/s"
        what = f"B={job.B} decode, KV lengths {min(job.L)}..{max(job.L)}"
        if cfg.get("ring"):
            what += ", sliding cache a ring of one window (512 rows)"
        vdef = "algorithmic K/V + q + out bytes of every layer's decode step / step time"
    elif isinstance(job, ProjJob):
        value, unit = job.M * steps * world / total, "tokens/s"
        what = (f"B={job.B} T={job.T} D={job.D}, " + ("q/k/v projection fused into the norm / RoPE / append"
                                                      if job.kind == "qkv" else
                                                      "o_proj + post-attention norm + residual"))
        vdef = "B*T tokens / step time (the fused projection of every layer)"
    else:
        value, unit = job.B * job.T * steps * world / total, "tokens/s"
        what = f"B={job.B} {'encoder (bidirectional)' if job.encoder else 'prefill'}, T={job.T}"
        vdef = "B*T tokens / step time (append + attention of every layer)"
    res = dict(workload=name, what=what + "; layers " + ", ".join(f"{r['layer_type']} hd {r['head_dim']}"
                                                                  for r in per_layer),
               value=value, unit=unit, value_definition=vdef, ms_per_step=total / steps * 1e3, steps=steps,
               rooflines=per_layer, clocks=clk, gpu_launches=job.launches_per_step() * steps,
               l2=f"flushed before every step ({L2_FLUSH_BYTES >> 20} MB write, outside the step's events)")
    del job, flush
    torch.cuda.empty_cache()
    return res


def _gpu_uuid(dev):
    import torch
    props = torch.cuda.get_device_properties(dev)
    u = str(getattr(props, "uuid", "") or "")
    if u and not u.startswith("GPU-"):
        u = "GPU-" + u
    return u


def run_layers(args, cfg):
    """`bench.py --workload <one- or two-layer workload>`: that workload's own line."""
    import torch
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dist_init("nccl")
    dev = torch.device("cuda", local)
    from gemma_dual_geometry_gb300 import build as g4build
    from gemma_dual_geometry_gb300 import g4attn as G
    g4build.build()
    G.lib()
    r = measure_layer_workload(args.workload, args, dev)
    dominant = max(r["rooflines"], key=lambda x: x["avg_launch_ms"])
    line = {"metric": METRIC, "value": r["value"], "unit": r["unit"], "n_gpus": world, "steps": r["steps"],
            "warmup": max(3, args.warmup), "ms_per_step": r["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), on device)",
            "config": {"workload": f"{args.workload}: {r['what']}", "l2": r["l2"],
                       "value_definition": r["value_definition"]},
            "roofline": dominant, "rooflines": r["rooflines"], "clocks": r["clocks"],
            "gpu_launches": r["gpu_launches"]}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(job, args, dev, world):
    """Prefill through the public API with the step's raw inputs copied in from
    pinned host memory and the last layer's output copied back, every step."""
    import torch
    host = []
    h2d = 0
    for x in job.X:
        hx = {}
        for k in ("q", "k", "v"):
            if k in x:
                h = torch.empty(x[k].shape, dtype=x[k].dtype, pin_memory=True)
                h.copy_(x[k])
                hx[k] = h
                h2d += h.numel() * h.element_size()
        host.append(hx)
    last_hd = job.st.geo[job.n - 1]["head_dim"]
    out_h = torch.empty(job.out[last_hd].shape, dtype=job.out[last_hd].dtype, pin_memory=True)
    d2h = out_h.numel() * out_h.element_size()
    steps = max(1, args.e2e_steps)
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    for _ in range(steps):
        for x, hx in zip(job.X, host):
            for k, h in hx.items():
                x[k].copy_(h, non_blocking=True)
        job.prefill()
        out_h.copy_(job.out[last_hd], non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    dt = reduce_max(e0.elapsed_time(e1) * 1e-3, dev)
    tokens = job.B * job.T * steps * world
    return {"value": tokens / dt, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "wall_s": wall, "what": "prefill of the 42-layer stack; inputs H2D from pinned host "
                                                     "memory and the last layer's output D2H inside the timed region"}


# ---------------------------------------------------------------- the oracle (CPU) arm
#
# The float64 oracle timed on all the host's cores on a bounded sample of the
# stack workload: sequence 0 of every layer, the append (norm / RoPE of q, k,
# v and the cache write) of a chunk of tokens, and attention for sampled query
# tokens (all heads) over the 4096-token cache.  The sample's arrays are built
# once (untimed) into .npy files that every worker maps; a spawn-context
# process pool (one single-threaded worker per core) runs the append of each
# layer, then the attention of (layer, query group) tasks.  Cost per token =
# append wall time / chunk + attention wall time / sampled queries; tokens/s
# is its inverse.

_ORACLE_MAPS = {}


def _oracle_arr(d, name, mode="r"):
    import numpy as np
    key = (d, name, mode)
    if key not in _ORACLE_MAPS:
        _ORACLE_MAPS[key] = np.load(os.path.join(d, name + ".npy"), mmap_mode=mode)
    return _ORACLE_MAPS[key]


def _oracle_task(task):
    """One timed unit of the sample in a pool worker: ("app", layer) or
    ("att", layer, first query, query count).  Returns seconds."""
    import numpy as np

    from oracle import g4_oracle as O
    d, spec = task[0], task[1]
    kind, l = task[2], task[3]
    g, src, T, H, Hkv = spec["geo"][l], spec["src"][l], spec["T"], spec["H"], spec["Hkv"]
    s_l = l if src < 0 else src
    lp = dict(g, kv_share_src=src)
    if kind == "app":
        q = _oracle_arr(d, f"q{l}")
        k = _oracle_arr(d, f"k{l}") if src < 0 else None
        v = _oracle_arr(d, f"v{l}") if src < 0 else None
        ck = _oracle_arr(d, f"ck{l}", "r+") if src < 0 else None
        cv = _oracle_arr(d, f"cv{l}", "r+") if src < 0 else None
        qw = _oracle_arr(d, f"qw{l}")
        kw = _oracle_arr(d, f"kw{l}") if src < 0 else None
        t0 = time.perf_counter()
        O.kv_append_normrope(lp, q, k, v, qw, kw, np.arange(q.shape[1])[None, :], ck, cv)
        return time.perf_counter() - t0
    q0, nq = task[4], task[5]
    qs = _oracle_arr(d, f"qs{l}")[:, q0:q0 + nq]
    tq = np.asarray(spec["tq"][q0:q0 + nq], dtype=np.int64)
    ck = _oracle_arr(d, f"ck{s_l}")
    cv = _oracle_arr(d, f"cv{s_l}")
    qw = _oracle_arr(d, f"qw{l}")
    t0 = time.perf_counter()
    qn = O.store(O.normrope_q(qs, qw, tq[None, :], g["head_dim"], g["theta"], g["rotary_fraction"], g["eps"]),
                 g["dtype"])
    rows = [(0, i, h) for i in range(nq) for h in range(H)]
    O.attention_rows(qn, ck, cv, rows, tq[None, :], [T], Hkv, g["layer_type"], g["window"], g["attn_scale"])
    return time.perf_counter() - t0


def oracle_worker(spec):
    """Runs in a subprocess (no GPU, one BLAS thread per process): builds the
    sample, then times it on a pool of one worker per core."""
    import multiprocessing as mp
    import shutil

    import numpy as np

    from gemma_dual_geometry_gb300 import workloads as W
    from oracle import g4_oracle as O

    cfg = W.CONFIGS[spec["workload"]]
    T, H, Hkv = cfg["T"], cfg["H"], cfg["Hkv"]
    n = len(cfg["types"])
    nq, chunk, group = spec["n_query"], spec["append_chunk"], spec["query_group"]
    is_s = [t == W.SLIDING for t in cfg["types"]]
    src = [O.kv_share_src(n, cfg["n_shared"], is_s, l) for l in range(n)]
    geo = [W.layer_geometry(cfg, l) for l in range(n)]
    tq = np.linspace(0, T - 1, nq).astype(np.int64)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    cores = max(1, min(cores, spec.get("max_cores") or cores))
    d = tempfile.mkdtemp(prefix="g4_oracle_sample_")

    def put(name, t):
        np.save(os.path.join(d, name + ".npy"), np.ascontiguousarray(t.double().numpy()))

    try:
        # setup (untimed): sequence 0's raw inputs for the appended chunk and
        # the sampled queries, and full-length caches of the owning layers
        # (seeded N(0,1) rows; the cost does not depend on the values)
        for l in range(n):
            x = W.layer_inputs(cfg, l, chunk, src[l] < 0, B=1)
            for k_, v_ in x.items():
                put({"q": "q", "k": "k", "v": "v", "q_norm_w": "qw", "k_norm_w": "kw"}[k_] + str(l), v_)
            put(f"qs{l}", W.normal((1, nq, H, geo[l]["head_dim"]), W.seed_for(cfg["seed"], l, 10), cfg["dtype"]))
            if src[l] < 0:
                ck, cv = W.prefilled_cache(cfg, l, T, B=1)
                put(f"ck{l}", ck)
                put(f"cv{l}", cv)
        sp = dict(geo=geo, src=src, T=T, H=H, Hkv=Hkv, tq=tq.tolist())
        app = [(d, sp, "app", l) for l in range(n)]
        att = [(d, sp, "att", l, q0, min(group, nq - q0)) for l in range(n) for q0 in range(0, nq, group)]
        # heaviest first (full layers, then sliding; owning layers' appends before q-only ones)
        app.sort(key=lambda t: -(geo[t[3]]["head_dim"] * (3 if src[t[3]] < 0 else 1)))
        att.sort(key=lambda t: -geo[t[3]]["head_dim"])
        steps = []
        with mp.get_context("spawn").Pool(cores) as pool:
            for _ in range(spec["warmup"] + spec["steps"]):
                t0 = time.perf_counter()
                t_app_cpu = sum(pool.map(_oracle_task, app, chunksize=1))
                t1 = time.perf_counter()
                t_att_cpu = sum(pool.map(_oracle_task, att, chunksize=1))
                t2 = time.perf_counter()
                steps.append(dict(t_append=t1 - t0, t_attn=t2 - t1, per_token_s=(t1 - t0) / chunk + (t2 - t1) / nq,
                                  cpu_s=t_app_cpu + t_att_cpu))
        return dict(steps=steps[spec["warmup"]:], cores=cores)
    finally:
        shutil.rmtree(d, ignore_errors=True)


def _oracle_subprocess(workload, steps, warmup, n_query=32, append_chunk=256, query_group=4, max_cores=None):
    spec = dict(workload=workload, steps=steps, warmup=warmup, n_query=n_query, append_chunk=append_chunk,
                query_group=query_group, max_cores=max_cores)
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    t0 = time.perf_counter()
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-worker", json.dumps(spec)],
                       capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("oracle worker failed: " + r.stderr[-2000:])
    res = json.loads(r.stdout.strip().splitlines()[-1])
    return res, time.perf_counter() - t0, spec


def _sample_text(spec, cores):
    return (f"sequence 0 of the stack: per layer, append of {spec['append_chunk']} tokens and attention for "
            f"{spec['n_query']} evenly spaced query tokens x 8 heads over the 4096-token cache; "
            f"tokens/s = 1 / (append wall s / token + attention wall s / query token); numpy float64 on a "
            f"spawn-context pool of {cores} single-threaded workers (one per host core), tasks = each layer's "
            f"append and (layer, group of {spec['query_group']} queries) attention")


def cpu_baseline(workload, steps=1, warmup=1):
    res, wall, spec = _oracle_subprocess(workload, steps, warmup)
    per = statistics.median(s["per_token_s"] for s in res["steps"])
    return {"value": 1.0 / per, "unit": "tokens/s", "cores": res["cores"], "kind": "oracle",
            "sample": _sample_text(spec, res["cores"]), "wall_s": wall,
            "cpu_s_per_step": statistics.median(s["cpu_s"] for s in res["steps"])}


def run_reference(args, cfg):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    res, wall, spec = _oracle_subprocess(args.workload, args.steps, args.warmup)
    per = [s["per_token_s"] for s in res["steps"]]
    value = 1.0 / statistics.median(per)
    step_s = statistics.mean(s["t_append"] + s["t_attn"] for s in res["steps"])
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1))",
        "config": {"workload": "attention-only 42-layer stack (5 sliding : 1 full, last 18 shared-KV), "
                               "n_heads 8, n_kv 2, head_dim 256 / global 512, window 512, batch 8, "
                               "prefill T=4096 then 128 decode steps", "global_batch": cfg["B"],
                   "seq_len": cfg["T"], "parallelism": f"host cores x{res['cores']}"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": res["cores"], "kind": "oracle",
                         "sample": "per step: " + _sample_text(spec, res["cores"])},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.oracle_worker:
        res = oracle_worker(json.loads(args.oracle_worker))
        print(json.dumps(res), flush=True)
        return
    from gemma_dual_geometry_gb300 import workloads as W
    cfg = W.CONFIGS[args.workload]
    if args.impl == "reference":
        run_reference(args, cfg)
    elif "decode_steps" in cfg:
        run_ours(args, cfg)
    else:
        run_layers(args, cfg)


if __name__ == "__main__":
    main()
