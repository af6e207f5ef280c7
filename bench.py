#!/usr/bin/env python
"""Benchmark of the W4A16 skinny GEMM on GB300: one JSON line on stdout.

Headline workload: the M=1 decode GEMV on (N=8192, K=8192) and (N=17408,
K=5120), group size 128, seeded synthetic inputs (X ~ N(0,1) in bf16, codes
uniform in [0,15], scales uniform in [0.005, 0.02]).  One step is one call of
w4a16_gemm per shape (the decode kernel plus, where the plan splits K, the
reduce kernel), with the weights marked resident (W4A16_FLAG_RESIDENT_WEIGHTS:
model weights written once, so a call may stream them into shared memory
while the kernel before it is still running).  Metric: algorithmic bytes (packed W + scales + X + Y) per
second, in GB/s.

Timing: W eager warm-up steps, then exactly K steps replayed from CUDA graphs
(one graph of K steps when K <= 2000, else graphs of G steps), bracketed by a
barrier and a synchronize, timed with CUDA events on the launching stream.
A device-side sleep kernel is queued just before the start event, so the
host has enqueued the graph launches by the time the start event fires and
the timed region holds the K steps back to back, not the host's launch
latency.  Each step uses the next of C weight copies whose total exceeds 4x
the L2 size, so every call streams its weights from HBM.  SM clocks and
throttle reasons are sampled with nvidia-smi during the timed region.

Also reported: the roofline of the dominant kernel (the decode kernel, timed
alone from a graph of back-to-back launches, so inter-launch gaps count
against it), an end-to-end figure through the public API with X copied in
from pinned host memory and Y copied back every step, per-shape figures for
every workload shape, and the CPU oracle's throughput on the host cores.

``--impl reference`` times the CPU oracle instead (the only reference this
method has), on a bounded sample of every step.  ``--shape M,N,K`` times one
GEMM shape the way the per-shape table does and prints that row only.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W4A16 GEMM TFLOP/s and HBM GB/s per shape (M=1 decode, M=1322 prefill) vs roofline"
HEADLINE_NAME = "decode_gemv"
HEADLINE_SHAPES = [(1, 8192, 8192), (1, 17408, 5120)]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--graph-steps", type=int, default=400, help="steps per captured CUDA graph")
    ap.add_argument("--no-shapes", action="store_true", help="skip the per-shape table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU baseline budget")
    ap.add_argument("--shape", type=str, default=None, metavar="M,N,K",
                    help="time one GEMM shape (graph of back-to-back calls) and print its row "
                         "only; 'grouped' times the grouped workload")
    ap.add_argument("--group-size", type=int, default=128, choices=[128, 64, 32],
                    help="scale group size G for --shape")
    ap.add_argument("--zero-points", action="store_true",
                    help="--shape: the zero-point variant (uint8 zero point per row and group)")
    return ap.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def workload_config():
    return {"workload": f"{HEADLINE_NAME}: M=1, (N=8192,K=8192) and (N=17408,K=5120), "
                        "group 128, int4 W x bf16 X, fp32 accumulate",
            "shapes": [list(s) for s in HEADLINE_SHAPES], "group_size": 128,
            "weights": "resident in HBM (W4A16_FLAG_RESIDENT_WEIGHTS: a call may start "
                       "streaming them before the previous kernel on the stream ends)"}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.25)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ distributed
def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(dist, seconds: float, device=None) -> float:
    """The slowest rank's time, returned on every rank (the whole job ends when
    its last replica ends).  dist None: one process."""
    if dist is None:
        return seconds
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, step_bytes: int, steps: int, seconds: float) -> float:
    """Whole-job throughput: every replica moves step_bytes per step."""
    return world * step_bytes * steps / seconds / 1e9


def maybe_init_dist(world, local):
    if world <= 1:
        return None
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local)
    dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return dist


# ---------------------------------------------------------------- our arm
class Shape:
    def __init__(self, torch, w4, syn, M, N, K, copies, device, seed=0, G=128, zp=False):
        inp = syn.make_gemm_inputs(M, N, K, G=G, seed=seed)
        self.torch = torch
        self.inp = inp
        self.M, self.N, self.K = M, N, K
        to_bf16 = lambda a: torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
        self.x = to_bf16(inp.x)
        # X rotates with the weights (a copy per weight copy), so no call finds
        # its activations in L2 either; end_to_end pins self.x instead.
        self.xs = [self.x] + [self.x.clone() for _ in range(copies - 1)]
        self.pin_x = False
        s = to_bf16(inp.scales)
        wp = w4.pack(torch.from_numpy(inp.w_canon.copy()).to(device))
        self.w = [wp] + [wp.clone() for _ in range(copies - 1)]
        self.s = [s] + [s.clone() for _ in range(copies - 1)]
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        self.z = None
        if zp:
            zd = torch.from_numpy(syn.make_zeros(N, K, G, seed=seed)).to(device)
            self.z = [zd] + [zd.clone() for _ in range(copies - 1)]
        self.plan = w4.plan(M, N, K, group_size=G, zero_points=zp)
        self.ws = torch.empty(max(self.plan["workspace_bytes"], 256), dtype=torch.uint8, device=device)
        self.launches = 1 + (1 if self.plan["split_k"] > 1 else 0)

    def xin(self, c):
        return self.x if self.pin_x else self.xs[c]

    def call(self, w4, i):
        c = i % len(self.w)
        w4.gemm(self.xin(c), self.w[c], self.s[c], out=self.y, workspace=self.ws, resident_weights=True,
                zeros=self.z[c] if self.z else None)

    def partials(self, w4, i):
        """The main kernel alone: the split-K decode kernel, or the whole call
        when the plan has one launch."""
        c = i % len(self.w)
        if self.plan["split_k"] == 1:
            return self.call(w4, i)
        return w4.gemm_partials(self.xin(c), self.w[c], self.s[c], out=self.y, workspace=self.ws,
                                resident_weights=True)

    def reduce(self, w4):
        sk = self.plan["split_k"]
        if sk > 1:
            parts = self.ws[: sk * self.M * self.N * 4].view(self.torch.float32)
            w4.splitk_reduce(parts.view(sk, self.M, self.N), out=self.y)


def copies_for(torch, device, bytes_per_copy):
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    return max(2, int(math.ceil(4.0 * l2 / max(bytes_per_copy, 1))))


def capture(torch, fn, n):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(0)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            fn(i)
    return g


def hide_launch_latency(torch, launches: int):
    """Queue a device-side sleep long enough for the host to enqueue
    `launches` graph launches behind it (about 20 us each), so that a start
    event recorded after it fires with the timed work already queued."""
    us = min(20000, 50 + 20 * launches)
    torch.cuda._sleep(int(us * 2000))        # cycles at about 2 GHz


def time_graph(torch, g, reps=1):
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    hide_launch_latency(torch, reps)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def our_arm(args, world, rank, local, dist):
    import torch
    import bf16_activation_quantized_gb300 as w4
    from bf16_activation_quantized_gb300 import build as build_mod
    from bf16_activation_quantized_gb300 import metrics
    from bf16_activation_quantized_gb300 import synthetic as syn

    build_mod.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    peaks, peaks_src = load_peaks()

    per_copy = sum(metrics.weight_bytes(N, K) for (_, N, K) in HEADLINE_SHAPES)
    C = copies_for(torch, device, per_copy)
    shapes = [Shape(torch, w4, syn, M, N, K, C, device) for (M, N, K) in HEADLINE_SHAPES]
    step_bytes = sum(metrics.algorithmic_bytes(s.M, s.N, s.K) for s in shapes)
    step_flops = sum(metrics.flops(s.M, s.N, s.K) for s in shapes)

    def step(i):
        for s in shapes:
            s.call(w4, i)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()

    # Up to 2000 steps are one graph of exactly K steps; longer runs replay
    # graphs of G steps (a multiple of the weight copies) and a remainder.
    if args.steps <= 2000:
        G = args.steps
    else:
        G = max(1, min(args.graph_steps, args.steps))
        G = max(C, (G // C) * C)
    full, rem = divmod(args.steps, G)
    g_full = capture(torch, step, G) if full else None
    g_rem = capture(torch, step, rem) if rem else None
    if g_full:
        g_full.replay()
    if g_rem:
        g_rem.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    hide_launch_latency(torch, full + (1 if g_rem else 0))
    e0.record()
    for _ in range(full):
        g_full.replay()
    if g_rem:
        g_rem.replay()
    e1.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    elapsed = max_over_ranks(dist, e0.elapsed_time(e1) / 1e3, device)
    value = whole_job_gbs(world, step_bytes, args.steps, elapsed)
    launches = args.steps * sum(s.launches for s in shapes)

    # Dominant kernel alone: graphs of back-to-back decode-kernel launches
    # (the whole call where the plan has one launch).
    R = max(C, (200 // C) * C)
    g_part = capture(torch, lambda i: [s.partials(w4, i) for s in shapes], R)
    t_part = min(time_graph(torch, g_part) for _ in range(3)) / R
    red_shapes = [s for s in shapes if s.plan["split_k"] > 1]
    t_red = 0.0
    if red_shapes:
        g_red = capture(torch, lambda i: [s.reduce(w4) for s in red_shapes], R)
        t_red = min(time_graph(torch, g_red) for _ in range(3)) / R
    achieved = step_bytes / t_part / 1e9
    peak_key = "hbm_gbs"
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks[peak_key],
                "unit": "GB/s", "frac": round(achieved / peaks[peak_key], 4),
                "traffic": load_traffic(),
                "kernel": ", ".join(sorted({("decode_rows_kernel (whole K, one launch)" if s.plan["whole_k"]
                                             else "decode_kernel (K slices) + splitk_reduce_kernel"
                                             if s.plan["split_k"] > 1 else "decode_kernel (K slices)")
                                            for s in shapes})) + " per shape per step",
                "kernel_us_per_step": round(t_part * 1e6, 3),
                "reduce_us_per_step": round(t_red * 1e6, 3),
                "peak_source": f"{peaks_src} (MEASURED_PEAKS.json hbm_gbs)" if peaks_src == "measured"
                else "fallback 6.8 TB/s"}

    # End to end through the public API: pinned X in, Y out, every step.
    e2e = end_to_end(torch, w4, shapes, min(args.steps, 2000), step_bytes)

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(elapsed / args.steps * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(), l2=f"weights rotate over {C} copies "
                       f"({C * per_copy / 1e6:.0f} MB > 4x L2) between steps",
                       parallelism=f"replicas x{world}", graph_steps=G,
                       plans=[s.plan for s in shapes]),
        "tflops": round(world * step_flops * args.steps / elapsed / 1e12, 4),
        "clocks": clocks, "e2e": e2e, "gpu_launches": launches, "roofline": roofline,
    }
    if rank == 0 and not args.no_shapes:
        out["per_shape"] = per_shape_table(torch, w4, syn, metrics, device, peaks,
                                           cpu=world == 1 and not args.no_cpu_baseline)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return out


def load_traffic():
    """DRAM bytes per step of the decode kernel from the committed ncu summary,
    or None when the kernel's sources changed after that capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        h = hashlib.sha256()
        for src in d["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != d["sources_sha256"]:
            return None
        return d.get("decode_gemv_bytes_per_step")
    except Exception:
        return None


def end_to_end(torch, w4, shapes, steps, step_bytes):
    """The step through the public API with host buffers: every step copies all
    of its X rows in from pinned host memory (one transfer: the shapes' X are
    views of one device buffer) and reads all of Y back (one transfer)."""
    dev = shapes[0].x.device
    xs = [s.M * s.K for s in shapes]
    ys = [s.M * s.N for s in shapes]
    dx = torch.empty(sum(xs), dtype=torch.bfloat16, device=dev)
    dy = torch.empty(sum(ys), dtype=torch.bfloat16, device=dev)
    saved = [(s.x, s.y) for s in shapes]
    ox = oy = 0
    for s, nx, ny in zip(shapes, xs, ys):     # offsets keep every X 16-byte aligned
        dx[ox:ox + nx].copy_(s.x.reshape(-1))
        s.x = dx[ox:ox + nx].view(s.M, s.K)
        s.pin_x = True
        s.y = dy[oy:oy + ny].view(s.M, s.N)
        ox += nx
        oy += ny
    hx = dx.cpu().pin_memory()
    hy = torch.empty(dy.shape, dtype=dy.dtype).pin_memory()
    h2d = hx.numel() * hx.element_size()
    d2h = hy.numel() * hy.element_size()

    def one(i):
        dx.copy_(hx, non_blocking=True)
        for s in shapes:
            s.call(w4, i)
        hy.copy_(dy, non_blocking=True)

    try:
        for i in range(3):
            one(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(steps):
            one(i)
        torch.cuda.synchronize()
        dt_eager = time.perf_counter() - t0

        # The same steps captured in CUDA graphs (as a serving loop replays its
        # decode step); the copies are inside the graph; wall clock.
        G = 100
        g = capture(torch, one, G)
        g.replay()
        torch.cuda.synchronize()
        reps = max(1, steps // G)
        t0 = time.perf_counter()
        for _ in range(reps):
            g.replay()
        torch.cuda.synchronize()
        dt_graph = (time.perf_counter() - t0) / (reps * G) * steps
        del g
    finally:
        for s, (x, y) in zip(shapes, saved):
            s.x, s.y = x, y
            s.pin_x = False
    return {"value": round(step_bytes * steps / dt_graph / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "eager_value": round(step_bytes * steps / dt_eager / 1e9, 1),
            "note": "wall clock; every step copies all X rows from pinned host memory (one "
                    "transfer) and reads all of Y back (one transfer); value: the steps "
                    "replayed from CUDA graphs of 100 captured steps (copies inside the graph); "
                    "eager_value: the same steps as eager Python calls; packed weights stay "
                    "resident"}


# Scale groups of 32 columns (the gfx1151 page benchmarks group_size=32) on a
# decode and a prefill shape; every other row uses groups of 128.
GROUP32_SHAPES = [("decode_gemv_g32", 1, 8192, 8192), ("decode_gemv_g32", 1, 17408, 5120),
                  ("prefill_g32", 1322, 19456, 2560), ("prefill_g32", 1322, 2560, 9728)]
# The zero-point variant (one uint8 zero point per row and scale group).
ZP_SHAPES = [("decode_gemv_zp", 1, 8192, 8192, 128), ("decode_gemv_zp", 1, 17408, 5120, 128),
             ("prefill_zp", 1322, 19456, 2560, 128), ("prefill_zp", 1322, 19456, 2560, 32)]


def oracle_sample_rate(compute_cols, N, nbytes, flops, budget_s=0.3):
    """The CPU oracle on a bounded sample of a row's work: compute_cols(c)
    computes output features [0, c) of every token; the time is scaled to the
    whole shape's algorithmic bytes and FLOPs (the oracle's work per feature is
    the same for every feature)."""
    import oracle
    c = max(1, N // 256)
    t0 = time.perf_counter()
    compute_cols(c)
    t = time.perf_counter() - t0
    want = min(N, max(1, int(c * budget_s / max(t, 1e-6))))
    if want > c:
        c = want
        t0 = time.perf_counter()
        compute_cols(c)
        t = time.perf_counter() - t0
    frac = c / N
    return {"value": round(nbytes * frac / t / 1e9, 4), "unit": "GB/s",
            "tflops": round(flops * frac / t / 1e12, 6), "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"output features [0, {c}) of {N} ({frac:.4f} of the shape), {t:.2f} s"}


def row_e2e(torch, w4, s, reps, nbytes, flops):
    """One shape through the public API with host buffers: every call copies X
    in from pinned host memory and Y back to it (wall clock, eager calls)."""
    hx = s.x.cpu().pin_memory()
    hy = torch.empty((s.M, s.N), dtype=torch.bfloat16).pin_memory()
    s.pin_x = True
    try:
        def one(i):
            s.x.copy_(hx, non_blocking=True)
            s.call(w4, i)
            hy.copy_(s.y, non_blocking=True)
        for i in range(3):
            one(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(reps):
            one(i)
        torch.cuda.synchronize()
        dt = (time.perf_counter() - t0) / reps
    finally:
        s.pin_x = False
    return {"value": round(nbytes / dt / 1e9, 1), "unit": "GB/s", "tflops": round(flops / dt / 1e12, 3),
            "h2d_bytes_per_call": int(hx.numel() * 2), "d2h_bytes_per_call": int(hy.numel() * 2),
            "calls": reps, "note": "wall clock, eager calls through w4a16_gemm; X copied in "
                                   "from pinned host memory and Y read back every call"}


def per_shape_table(torch, w4, syn, metrics, device, peaks, only=None, group_size=128, zp=False,
                    cpu=True):
    shapes = [("tiny", 4, 256, 512, 128, False)]
    for name, lst in (("decode_gemv", syn.WORKLOADS["decode_gemv"]),
                      ("decode_sweep_gate_up", syn.WORKLOADS["decode_sweep_gate_up"]),
                      ("decode_sweep_down", syn.WORKLOADS["decode_sweep_down"]),
                      ("prefill", syn.WORKLOADS["prefill"]),
                      ("prefill_long", syn.WORKLOADS["prefill_long"])):
        shapes += [(name, M, N, K, 128, False) for (M, N, K) in lst]
    shapes += [(name, M, N, K, 32, False) for (name, M, N, K) in GROUP32_SHAPES]
    shapes += [(name, M, N, K, G, True) for (name, M, N, K, G) in ZP_SHAPES]
    if only is not None:
        if len(only) == 4:    # G, M_total, N, K: the grouped workload
            return [grouped_row(torch, w4, syn, metrics, device, peaks)]
        named = [sh for sh in shapes if sh[1:] == tuple(only) + (group_size, zp)]
        shapes = named[:1] or [("custom",) + tuple(only) + (group_size, zp)]
    rows = []
    for name, M, N, K, G, with_zp in shapes:
        # (zero points: one more byte per row and scale group)
        wb = metrics.weight_bytes(N, K, G) + (N * (K // G) if with_zp else 0)
        C = copies_for(torch, device, wb + 2 * M * K)
        s = Shape(torch, w4, syn, M, N, K, C, device, G=G, zp=with_zp)
        R = max(C, (100 // C) * C) if M < 512 else C
        g = capture(torch, lambda i: s.call(w4, i), R)
        g.replay()
        t = statistics.median(time_graph(torch, g) for _ in range(5)) / R
        nbytes = metrics.algorithmic_bytes(M, N, K, G) + (N * (K // G) if with_zp else 0)
        fl = metrics.flops(M, N, K)
        t_roof = metrics.roofline_seconds(fl, nbytes, peaks["bf16_tflops"] * 1e12, peaks["hbm_gbs"] * 1e9)
        row = {"workload": name, "M": M, "N": N, "K": K, "group_size": G, "zero_points": with_zp,
               "us": round(t * 1e6, 3),
               "tflops": round(fl / t / 1e12, 3), "gbs": round(nbytes / t / 1e9, 1),
               "roofline_frac": round(t_roof / t, 4),
               "bound": "hbm" if nbytes / (peaks["hbm_gbs"] * 1e9) >= fl / (peaks["bf16_tflops"] * 1e12) else "tensor",
               "arm": s.plan["arm"], "split_k": s.plan["split_k"], "whole_k": s.plan["whole_k"],
               "copies": C}
        if name == "prefill":
            row["e2e"] = row_e2e(torch, w4, s, 20, nbytes, fl)
        if cpu:
            import oracle
            inp = s.inp
            if with_zp:
                zc = syn.make_zeros(N, K, G, seed=0)
                fn = lambda c: oracle.gemm_zp(inp.x, inp.w_canon[:c], inp.scales[:c], zc[:c], M, c, K, G=G)
            else:
                fn = lambda c: oracle.gemm(inp.x, inp.w_canon[:c], inp.scales[:c], M, c, K, G=G)
            row["cpu_baseline"] = oracle_sample_rate(fn, N, nbytes, fl)
        rows.append(row)
        del g, s
        torch.cuda.empty_cache()
    if only is None:
        rows.append(grouped_row(torch, w4, syn, metrics, device, peaks, cpu))
        for B, M, N, K in BATCHED_SHAPES:
            rows.append(batched_row(torch, w4, syn, metrics, device, peaks, B, M, N, K, cpu))
    return rows


# The batched op's report rows: the shapes of the pages' batched table (B
# independent products of one shape, one launch).
BATCHED_SHAPES = [(4, 128, 8192, 3584), (2, 2048, 7168, 8192)]


def batched_row(torch, w4, syn, metrics, device, peaks, B, M, N, K, cpu=True):
    inps = [syn.make_gemm_inputs(M, N, K, seed=b) for b in range(B)]
    bits = lambda a: torch.from_numpy(a.view("int16").copy()).view(torch.bfloat16).to(device)
    x = torch.stack([bits(i.x) for i in inps])
    s = torch.stack([bits(i.scales) for i in inps])
    w = torch.stack([w4.pack(torch.from_numpy(i.w_canon.copy()).to(device)) for i in inps])
    y = torch.empty((B, M, N), dtype=torch.bfloat16, device=device)
    C = copies_for(torch, device, B * metrics.weight_bytes(N, K))
    ws = [w] + [w.clone() for _ in range(C - 1)]
    plan = w4.plan_batched(B, M, N, K)
    R = max(C, (20 // C) * C)
    g = capture(torch, lambda i: w4.gemm_batched(x, ws[i % C], s, out=y, resident_weights=True), R)
    g.replay()
    t = statistics.median(time_graph(torch, g) for _ in range(3)) / R
    nbytes = B * metrics.algorithmic_bytes(M, N, K)
    fl = B * metrics.flops(M, N, K)
    t_roof = metrics.roofline_seconds(fl, nbytes, peaks["bf16_tflops"] * 1e12, peaks["hbm_gbs"] * 1e9)
    row = {"workload": "batched", "batch": B, "M": M, "N": N, "K": K,
           "us": round(t * 1e6, 3), "tflops": round(fl / t / 1e12, 3), "gbs": round(nbytes / t / 1e9, 1),
           "roofline_frac": round(t_roof / t, 4),
           "bound": "hbm" if nbytes / (peaks["hbm_gbs"] * 1e9) >= fl / (peaks["bf16_tflops"] * 1e12) else "tensor",
           "arm": plan["arm"], "split_k": plan["split_k"], "copies": C}
    if cpu:
        import oracle
        row["cpu_baseline"] = oracle_sample_rate(
            lambda c: [oracle.gemm(i.x, i.w_canon[:c], i.scales[:c], M, c, K) for i in inps],
            N, nbytes, fl)
    del g, ws
    torch.cuda.empty_cache()
    return row


def grouped_row(torch, w4, syn, metrics, device, peaks, cpu=True):
    """The grouped workload: one launch over all groups, sizes read on the device."""
    G, MT, N, K = (syn.GROUPED_WORKLOAD[k] for k in ("num_groups", "M_total", "N", "K"))
    inp = syn.make_grouped_inputs(G, MT, N, K, seed=0)
    bits = lambda a: torch.from_numpy(a.view("int16").copy()).view(torch.bfloat16).to(device)
    x = bits(inp.x)
    s = bits(inp.scales)
    w = torch.stack([w4.pack(torch.from_numpy(inp.w_canon[g].copy()).to(device)) for g in range(G)])
    sizes = torch.from_numpy(inp.m_sizes.copy()).to(device)
    y = torch.empty((MT, N), dtype=torch.bfloat16, device=device)
    _, st = w4.gemm_grouped(x, w, s, sizes, out=y)      # sizes the status word once
    torch.cuda.synchronize()
    C = copies_for(torch, device, G * metrics.weight_bytes(N, K))
    ws = [w] + [w.clone() for _ in range(C - 1)]
    R = max(C, (40 // C) * C)
    g = capture(torch, lambda i: w4.gemm_grouped(x, ws[i % C], s, sizes, out=y, status=st), R)
    g.replay()
    t = statistics.median(time_graph(torch, g) for _ in range(5)) / R
    nbytes = metrics.grouped_algorithmic_bytes(G, MT, N, K)
    fl = metrics.flops(MT, N, K)
    t_roof = metrics.roofline_seconds(fl, nbytes, peaks["bf16_tflops"] * 1e12, peaks["hbm_gbs"] * 1e9)
    row = {"workload": "grouped", "M": MT, "N": N, "K": K, "groups": G,
           "us": round(t * 1e6, 3), "tflops": round(fl / t / 1e12, 3), "gbs": round(nbytes / t / 1e9, 1),
           "roofline_frac": round(t_roof / t, 4), "bound": "tensor", "arm": "tensor (grouped)",
           "split_k": 1, "copies": C}
    if cpu:
        import oracle
        row["cpu_baseline"] = oracle_sample_rate(
            lambda c: oracle.gemm_grouped(inp.x, inp.w_canon[:, :c], inp.scales[:, :c], inp.m_sizes,
                                          MT, c, K), N, nbytes, fl)
    del g, ws
    torch.cuda.empty_cache()
    return row


# ----------------------------------------------------------- CPU baseline
def cpu_baseline(budget_s: float, shapes=HEADLINE_SHAPES, frac=1.0):
    """The oracle on the host cores: whole steps of the headline workload (or a
    column slice of each shape when frac < 1), repeated until budget_s."""
    import oracle
    from bf16_activation_quantized_gb300 import metrics
    from bf16_activation_quantized_gb300 import synthetic as syn
    inps = [syn.make_gemm_inputs(M, N, K, seed=0) for (M, N, K) in shapes]
    cols = [max(1, int(round(i.N * frac))) for i in inps]
    nbytes = sum(metrics.algorithmic_bytes(i.M, c, i.K) for i, c in zip(inps, cols))
    reps, t_total = 0, 0.0
    while reps == 0 or t_total < budget_s:
        t0 = time.perf_counter()
        for i, c in zip(inps, cols):
            oracle.gemm_cols(i.x, i.w_canon, i.scales, i.M, i.N, i.K, 0, c)
        t_total += time.perf_counter() - t0
        reps += 1
    per_step = t_total / reps
    sample = ("whole headline steps (both shapes, all outputs)" if frac >= 1 else
              f"output features [0, {cols}) of each shape, i.e. {frac:.4f} of every step")
    return {"value": round(nbytes / per_step / 1e9, 4), "unit": "GB/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{sample}; {reps} repetitions, {t_total:.1f} s",
            "s_per_step": per_step}


def reference_arm(args, world, rank):
    """The CPU oracle timed on the headline workload: each step is a bounded
    column sample of both shapes so that warm-up + steps finish in minutes."""
    import oracle
    from bf16_activation_quantized_gb300 import metrics
    from bf16_activation_quantized_gb300 import synthetic as syn
    inps = [syn.make_gemm_inputs(M, N, K, seed=0) for (M, N, K) in HEADLINE_SHAPES]
    # calibrate on 1/64 of the outputs
    t0 = time.perf_counter()
    for i in inps:
        oracle.gemm_cols(i.x, i.w_canon, i.scales, i.M, i.N, i.K, 0, max(1, i.N // 64))
    t_cal = (time.perf_counter() - t0) * 64
    budget = 150.0 / max(1, args.steps + args.warmup)
    frac = min(1.0, budget / max(t_cal, 1e-9))
    cols = [max(1, int(round(i.N * frac))) for i in inps]
    nbytes = sum(metrics.algorithmic_bytes(i.M, c, i.K) for i, c in zip(inps, cols))

    def one():
        for i, c in zip(inps, cols):
            oracle.gemm_cols(i.x, i.w_canon, i.scales, i.M, i.N, i.K, 0, c)

    for _ in range(max(3, args.warmup)):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - t0
    value = nbytes * args.steps / dt / 1e9
    sample = f"output features [0, {cols}) of each shape per step ({frac:.5f} of the step's work)"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(dt / args.steps * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_info()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(reference_arm(args, world, rank)), flush=True)
        return 0
    if args.shape:
        import torch
        import bf16_activation_quantized_gb300 as w4
        from bf16_activation_quantized_gb300 import build as build_mod
        from bf16_activation_quantized_gb300 import metrics
        from bf16_activation_quantized_gb300 import synthetic as syn
        build_mod.build()
        device = torch.device("cuda", local)
        torch.cuda.set_device(device)
        peaks, _ = load_peaks()
        only = ([0, 0, 0, 0] if args.shape == "grouped" else
                [int(v) for v in args.shape.split(",")])
        if rank == 0:
            print(json.dumps(per_shape_table(torch, w4, syn, metrics, device, peaks, only,
                                             args.group_size, args.zero_points,
                                             cpu=not args.no_cpu_baseline)[0]), flush=True)
        return 0
    dist = maybe_init_dist(world, local)
    out = our_arm(args, world, rank, local, dist)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
