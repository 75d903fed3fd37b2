#!/usr/bin/env python
"""Benchmark of the bwgemm hot path: dense C = A * B^T in bf16 on one GB300.

One step = one pass of the whole path over one batch of synthetic input:
plan lookup + TMA descriptors on the host, then one launch of the
persistent tcgen05 kernel (producer / MMA / epilogue, split-K where the shape
asks for it).  The headline workload is the 4096^3 square GEMM with
N(0,1)/sqrt(K) bf16 operands; the pages' Llama-3-70B prefill and decode
linears, the fp16 square and the tail shapes are timed alongside and
reported under "shapes".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: CUDA events on the launching stream.  The GPU idles ``--idle``
seconds, then W untimed warm-up steps run straight into the K timed steps,
which are bracketed by a device synchronisation on both sides (so every box
starts the timed region from the same state; cuBLAS's context figure is timed
the same way).  ``value`` is the K steps' mean; ``median_ms`` is the median of
at least 50 separately event-timed launches.  Inputs rotate
over enough copies that their total exceeds twice the L2 (129 MB), so no step
reads operands left in L2 by the step before.  The library runs on one GPU
and has no multi-GPU path: ``--gpus`` other than 1 is refused.

The JSON line ends with ``shapes``, a compact summary of every other page
shape (microseconds per launch, fraction of its roofline, cuBLAS on the same
tensors), so that it survives in a short tail of the output; the full
per-shape records go to stderr.

``--impl reference`` times the CPU oracle (the plain fp64 triple loop) on the
host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "bf16 GEMM TFLOP/s + % of GB300 dense roofline (4096³, prefill, M=256 decode)"
HEADLINE = "square4096"
EXTRA_SHAPES = ["square4096_fp16", "prefill_attn_out", "prefill_mlp_up", "decode_attn_out",
                "decode_qkv", "decode_mlp_up", "decode_mlp_down", "gemma_512x8192x5376",
                "tail_m1", "tail_m16", "tail_m64", "tail_m200"]
PAGES_4096_BF16 = 1772.9  # TFLOP/s, the Blackwell deep dive's final kernel, on B200
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["gemm_kernel.cuh", "ptx.cuh", "kernel_params.h", "gemm_sm103.cu", "planner.cpp",
                  "api.cpp", "internal.h", "skinny_kernel.cuh", "skinny_sm103.cu", "wholek_kernel.cuh",
                  "wholek_sm103.cu"]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "dense_gemm_blackwell_03_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash()
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if len(line) >= 3 and line[0] == want and line[1] == workload:
                return int(line[2])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs.

    Samples count as "under load" when nvidia-smi's own timestamp falls inside
    the wall-clock window bracketed by begin() / end() around the timed region
    (utilization.gpu is a trailing average and lags a sub-second region)."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.device_index = device_index
        self.window = None
        self._t0 = None
        self.rows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.device_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def begin(self):
        self._t0 = datetime.datetime.now()

    def end(self):
        if self._t0 is not None:
            self.window = (self._t0, datetime.datetime.now())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 11:
                continue
            try:
                when = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                when = None
            try:
                rows.append({"t": when, "sm": float(parts[2]), "max": float(parts[3]),
                             "power": float(parts[4]) if parts[4] not in ("", "[N/A]") else None,
                             "hw": parts[7], "hw_thermal": parts[8], "sw_thermal": parts[9],
                             "power_cap": parts[10]})
            except ValueError:
                continue
        self.rows = rows
        return self.summary(self.window)

    def summary(self, window):
        """Clock / throttle summary of the samples timestamped inside `window`
        (a (start, end) pair of datetimes; all samples if none fall inside)."""
        rows = self.rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        in_window = []
        if window:
            lo, hi = window
            in_window = [r for r in rows if r["t"] is not None and lo <= r["t"] <= hi]
        loaded = in_window or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("power_cap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        powers = [r["power"] for r in loaded if r["power"] is not None]
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(in_window),
                "power_w_median": statistics.median(powers) if powers else None,
                "selection": ("samples timestamped inside the timed region" if in_window else
                              "all samples (none fell inside the timed region)")}


def input_sets(shape, device, l2_bytes, max_sets=4):
    """Enough seeded copies of (A, B, C) that consecutive steps never find
    their operands in L2."""
    import torch
    from dense_gemm_blackwell_03_gb300.workloads import make_inputs, TORCH_DTYPES
    set_bytes = shape.algorithmic_bytes
    n = 1 if set_bytes >= 2 * l2_bytes else min(max_sets, math.ceil(3 * l2_bytes / set_bytes))
    sets = []
    for i in range(max(n, 1)):
        A, B = make_inputs(shape, device=device, seed=None if i == 0 else 7919 * i + 17)
        C = torch.empty((shape.M, shape.N), dtype=TORCH_DTYPES[shape.dtype], device=device)
        sets.append((A, B, C))
    return sets


def time_region(fn, sets, steps, warmup, stream):
    """Run fn(A, B, C) `steps` times back to back (rotating input sets) between
    two events on the launching stream, bracketed by a device synchronisation
    on both sides; return the elapsed milliseconds."""
    import torch
    for i in range(warmup):
        fn(*sets[i % len(sets)])
    torch.cuda.synchronize()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_begin.record(stream)
    for i in range(steps):
        fn(*sets[i % len(sets)])
    t_end.record(stream)
    torch.cuda.synchronize()
    return t_begin.elapsed_time(t_end)


def time_each(fn, sets, iters, stream):
    """Per-iteration event times (ms) for the median / percentiles: each
    iteration is bracketed by its own pair of events."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(iters)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(iters)]
    torch.cuda.synchronize()
    for i in range(iters):
        starts[i].record(stream)
        fn(*sets[i % len(sets)])
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def time_graph(fn, sets, launches, per_graph=20):
    """Milliseconds per launch with the host out of the loop: `per_graph`
    launches (rotating input sets) captured once in a CUDA graph on the
    current stream, the graph replayed back to back between two events.  For
    launches of a few tens of microseconds the host's cost per call (Python,
    argument checks, the driver) is close to the GPU's time, so back-to-back
    eager launches can measure the host; both arms are timed this way too."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(3):
            fn(*sets[i % len(sets)])
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(per_graph):
            fn(*sets[i % len(sets)])
    replays = max(3, launches // per_graph)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(replays):
        g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (replays * per_graph)
    del g
    return ms


SUSTAINED_REGION_S = 0.5  # timed regions at least this long run under the power cap


def tensor_peak_regime(region_seconds: float) -> str:
    """Which measured tensor peak a timed region of back-to-back launches is
    held to: the sustained one (measured over seconds under the power cap)
    once the region lasts SUSTAINED_REGION_S or longer, else the burst one."""
    return "sustained" if region_seconds >= SUSTAINED_REGION_S else "burst"


def aggregate(seconds: float, work_per_step: float, steps: int):
    """Throughput of one GPU's timed region.  Returns (seconds, work_per_second)."""
    return seconds, work_per_step * steps / seconds


def compact_shape(rec: dict) -> dict:
    """The short form of one shape's record that ends the JSON line: time per
    launch (us), fraction of its roofline keyed by the bound ("hbm" or
    "tensor"), cuBLAS's time on the same tensors (cb_us), both again under
    CUDA graph replay (g_us, cb_g_us) and the median SM clock while it ran."""
    r = rec["roofline"]
    out = {"us": rec["us"], r["bound"]: r["frac"], "cb_us": rec.get("cublas_us")}
    if rec.get("graph_us") is not None:
        out["g_us"] = rec["graph_us"]
        out["cb_g_us"] = rec.get("cublas_graph_us")
    mhz = (rec.get("clocks") or {}).get("sm_mhz")
    if mhz is not None:
        out["mhz"] = int(mhz)
    return out


def roofline_entry(shape, seconds, peaks):
    """Bound, achieved and peak for one shape (the min(peak, AI x BW) roofline)."""
    flops = shape.flops
    nbytes = shape.algorithmic_bytes
    ai = flops / nbytes
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    tflops = flops / seconds / 1e12
    gbs = nbytes / seconds / 1e9
    attainable = min(peaks["bf16_tflops"], ai * peaks["hbm_gbs"] / 1e3)
    if ai >= ridge:
        return {"bound": "tensor", "achieved": round(tflops, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(tflops / peaks["bf16_tflops"], 4),
                "roofline_frac": round(tflops / attainable, 4), "ai_flop_per_byte": round(ai, 1)}
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / peaks["hbm_gbs"], 4), "roofline_frac": round(tflops / attainable, 4),
            "ai_flop_per_byte": round(ai, 1), "tflops": round(tflops, 1)}


def cpu_baseline(shape, target_s=12.0):
    """The oracle as it stands, on the host cores, on a bounded sample of rows."""
    import oracle
    from dense_gemm_blackwell_03_gb300.workloads import bits_of, make_inputs
    A, B = make_inputs(shape, device="cpu")
    a, b = bits_of(A), bits_of(B)
    threads = oracle.max_threads()
    probe = min(shape.M, max(threads, 8))
    t0 = time.perf_counter()
    oracle.gemm(a, b, shape.dtype, rows=list(range(probe)))
    rate = probe / (time.perf_counter() - t0)
    rows = int(min(shape.M, max(probe, rate * target_s)))
    sel = list(range(0, shape.M, max(1, shape.M // rows)))[:rows]
    t0 = time.perf_counter()
    oracle.gemm(a, b, shape.dtype, rows=sel)
    dt = time.perf_counter() - t0
    flops = 2.0 * len(sel) * shape.N * shape.K
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{len(sel)} of {shape.M} rows of C ({len(sel)}x{shape.N}x{shape.K}, "
                      f"fp64 triple loop, {dt:.1f} s on {threads} threads); "
                      f"TFLOP/s extrapolated per row to the full {shape.M}x{shape.N}x{shape.K}"}


def run_reference(args):
    """--impl reference: the CPU oracle timed step by step on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:  # one line from rank 0 only, should a launcher start several
        return 0
    import oracle
    from dense_gemm_blackwell_03_gb300.workloads import SHAPES, bits_of, make_inputs
    shape = SHAPES[args.shape]
    A, B = make_inputs(shape, device="cpu")
    a, b = bits_of(A), bits_of(B)
    threads = oracle.max_threads()
    # size each step so that warm-up + timed steps take about args.ref_budget seconds
    t0 = time.perf_counter()
    oracle.gemm(a, b, shape.dtype, rows=list(range(min(shape.M, threads))))
    per_output = (time.perf_counter() - t0) / (min(shape.M, threads) * shape.N)
    outputs = max(threads, int(args.ref_budget / (args.steps + args.warmup) / per_output))
    # rows spread over all threads (the oracle parallelises over rows of C)
    if outputs >= threads * shape.N:
        nrows, ncols = min(shape.M, outputs // shape.N), None
    else:
        nrows = min(shape.M, threads)
        ncols = list(range(max(1, min(shape.N, outputs // nrows))))
    rows = list(range(nrows))
    for _ in range(args.warmup):
        oracle.gemm(a, b, shape.dtype, rows=rows, cols=ncols)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.gemm(a, b, shape.dtype, rows=rows, cols=ncols)
        times.append(time.perf_counter() - t0)
    n_out = nrows * (len(ncols) if ncols else shape.N)
    flops = 2.0 * n_out * shape.K
    mean = sum(times) / len(times)
    value = flops / mean / 1e12
    sample = (f"{n_out} outputs of C per step ({nrows} row(s) x "
              f"{len(ncols) if ncols else shape.N} cols, K={shape.K}), fp64 triple loop")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(mean * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{shape.name}: C=A*B^T, M={shape.M} N={shape.N} K={shape.K}, "
                               f"{shape.dtype} in/out", "M": shape.M, "N": shape.N, "K": shape.K},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    from dense_gemm_blackwell_03_gb300 import binding
    from dense_gemm_blackwell_03_gb300.workloads import SHAPES, TORCH_DTYPES, make_inputs

    local_rank = 0  # the one GPU this runs on
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)

    binding.load_library(build_if_missing=True)
    peaks = load_peaks()
    props = torch.cuda.get_device_properties(device)
    l2_bytes = int(getattr(props, "L2_cache_size", 129 * 10 ** 6)) or 129 * 10 ** 6
    shape = SHAPES[args.shape]
    stream = torch.cuda.current_stream(device)
    plan = binding.Plan(local_rank)

    def ours(A, B, C):
        plan.gemm(A, B, out=C, stream=stream)

    sets = input_sets(shape, device, l2_bytes)
    ours(*sets[0])  # the plan's tensor maps and the module, set up outside the region
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    # Every box starts from the same state: the GPU idles, then the W warm-up
    # steps run straight into the K timed ones (cuBLAS below the same way).
    time.sleep(args.idle)
    for i in range(args.warmup):
        ours(*sets[i % len(sets)])
    torch.cuda.synchronize()
    n0 = plan.launch_count()
    sampler.begin()
    total_ms = time_region(ours, sets, args.steps, 0, stream)
    sampler.end()
    clocks = sampler.stop()
    launches = plan.launch_count() - n0
    st = plan.status(stream)
    if st != 0:
        raise SystemExit(f"device status {st} after the timed region")
    kcfg = plan.last_config()
    per = time_each(ours, sets, max(50, min(args.steps, 200)), stream)

    total_s, flops_per_s = aggregate(total_ms / 1e3, shape.flops, args.steps)
    ms_per_step = total_s * 1e3 / args.steps
    value = flops_per_s / 1e12
    per_sorted = sorted(per)
    median_ms = statistics.median(per)
    avg_launch_s = total_s / args.steps  # one kernel launch per step, back to back

    # The measured tensor peak has a burst figure (cuBLAS timed briefly) and a
    # sustained one (seconds of back-to-back GEMMs under the power cap); the
    # timed region takes the one that matches its own length, and reports its
    # fraction of the other beside it.
    regime = tensor_peak_regime(total_s)
    tensor_peak = peaks["bf16_tflops_sustained"] if regime == "sustained" else peaks["bf16_tflops"]
    roof = roofline_entry(shape, avg_launch_s, dict(peaks, bf16_tflops=tensor_peak))
    roofline = {"bound": roof["bound"], "achieved": roof["achieved"], "peak": roof["peak"],
                "unit": roof["unit"], "frac": roof["frac"],
                "frac_of_burst_peak": (round(roof["achieved"] / peaks["bf16_tflops"], 4)
                                       if roof["bound"] == "tensor" else None),
                "frac_of_sustained_peak": (round(roof["achieved"] / peaks["bf16_tflops_sustained"], 4)
                                           if roof["bound"] == "tensor" else None),
                "traffic": recorded_traffic(shape.name),
                "peak_source": (f"{peaks['source']} ({regime} cuBLAS bf16: timed region {total_s * 1e3:.1f} ms)"
                                if roof["bound"] == "tensor" else f"{peaks['source']} (copy bandwidth)"),
                "kernel": "bwgemm::gemm_kernel (persistent tcgen05)",
                "algorithmic": (f"{shape.flops / 1e9:.1f} GFLOP per launch (2MNK)"
                                if roof["bound"] == "tensor" else
                                f"{shape.algorithmic_bytes / 1e6:.1f} MB per launch")}

    # cuBLAS (torch.matmul) on the same tensors, as same-box context
    def cublas(A, B, C):
        torch.matmul(A, B.t(), out=C)
    torch.cuda.synchronize()
    time.sleep(args.idle)
    cb_ms = time_region(cublas, sets, args.steps, args.warmup, stream)
    cb_s = cb_ms / 1e3 / args.steps

    # end-to-end through the C ABI with host buffers (H2D of A, B and D2H of C each step)
    e2e = None
    if not args.no_e2e:
        A0, B0, _ = sets[0]
        hA = A0.cpu().pin_memory()
        hB = B0.cpu().pin_memory()
        hC = torch.empty((shape.M, shape.N), dtype=TORCH_DTYPES[shape.dtype]).pin_memory()
        for _ in range(3):
            plan.gemm_host(hA, hB, out=hC, stream=stream)
        e2e_steps = max(5, min(args.steps, 30))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            plan.gemm_host(hA, hB, out=hC, stream=stream)
        e2e_s, e2e_flops = aggregate(time.perf_counter() - t0, shape.flops, e2e_steps)
        e2e = {"value": round(e2e_flops / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": 2 * (shape.M * shape.K + shape.N * shape.K),
               "d2h_bytes_per_step": 2 * shape.M * shape.N, "steps": e2e_steps,
               "api": "bwgemm_run_host (pinned host A, B, C)"}

    # the pages' other shapes, timed alongside (not the headline)
    shapes = {}
    if not args.no_extra:
        def steady(fn, ssets):
            """Seconds per step and the wall-clock window of the timed blocks.
            Each shape is timed in its own steady state: the GPU first idles for
            `cooldown` seconds, so that no shape starts from the power-capped
            clocks of the one before it; then the shape itself runs for about
            `shape_warmup` seconds, long enough for the clock and power
            controller to settle on its load (a dense-GEMM loop started after
            idle first overshoots the power cap and is throttled harder than
            in its steady state); then the median of three timed blocks of
            about 0.1 s is taken."""
            torch.cuda.synchronize()
            time.sleep(args.cooldown)
            pilot = time_region(fn, ssets, 10, 5, stream) / 1e3 / 10
            it = int(min(5000, max(50, 0.1 / max(pilot, 1e-7))))
            for _ in range(max(1, round(args.shape_warmup / 0.1))):
                time_region(fn, ssets, it, 0, stream)
            t0 = datetime.datetime.now()
            per = statistics.median(time_region(fn, ssets, it, 0, stream) / 1e3 / it for _ in range(3))
            return per, (t0, datetime.datetime.now())

        xsampler = ClockSampler(local_rank)
        xsampler.start()
        windows = {}

        extra = [SHAPES[n] for n in EXTRA_SHAPES]
        if args.fp16_extra:
            # the same shapes in fp16 (inputs rounded from the same fp32 draws)
            extra += [SHAPES[n].with_dtype("fp16") for n in EXTRA_SHAPES if SHAPES[n].dtype != "fp16"]
        for s in extra:
            name = s.name
            ssets = input_sets(s, device, l2_bytes, max_sets=3)
            t, windows[name] = steady(ours, ssets)
            if plan.status(stream) != 0:
                raise SystemExit(f"device status error on {name}")
            cfg = plan.last_config()
            med = statistics.median(time_each(ours, ssets, 50, stream)) / 1e3
            # both arms also with the host out of the loop (CUDA graph replay,
            # launches on the capturing stream), median of three timings
            n_g = int(min(2000, max(60, 0.05 / max(t, 1e-7))))
            g_ours = statistics.median(
                time_graph(lambda A, B, C: plan.gemm(A, B, out=C), ssets, n_g) for _ in range(3)) / 1e3
            t_cb, _ = steady(cublas, ssets)
            g_cb = statistics.median(time_graph(cublas, ssets, n_g) for _ in range(3)) / 1e3
            r = roofline_entry(s, t, peaks)
            shapes[name] = {"M": s.M, "N": s.N, "K": s.K, "dtype": s.dtype,
                            "us": round(t * 1e6, 2), "median_us": round(med * 1e6, 2),
                            "tflops": round(s.flops / t / 1e12, 1),
                            "gbs": round(s.algorithmic_bytes / t / 1e9, 1),
                            "roofline": r,
                            "cublas_us": round(t_cb * 1e6, 2),
                            "cublas_tflops": round(s.flops / t_cb / 1e12, 1),
                            "graph_us": round(g_ours * 1e6, 2),
                            "cublas_graph_us": round(g_cb * 1e6, 2),
                            "kernel_config": {k: cfg[k] for k in ("variant", "tile_m", "tile_n",
                                                                  "split_k", "schedule", "grid")}}
            del ssets
            torch.cuda.empty_cache()
        xsampler.stop()
        for name, win in windows.items():
            c = xsampler.summary(win)
            shapes[name]["clocks"] = {"sm_mhz": c["sm_mhz"], "reasons": c["reasons"],
                                      "samples_under_load": c.get("samples_under_load", 0)}

    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(shape, target_s=args.cpu_seconds)

    # The nominal dense peak from a measured per-SM tensor rate (a tcgen05.mma
    # probe timed in SM cycles) x SMs x the maximum SM clock; the fraction
    # against it is printed beside the one against the measured cuBLAS peak.
    if roof["bound"] == "tensor":
        try:
            rate, sms = binding.probe_tensor_rate(local_rank)
            max_mhz = clocks.get("sm_max_mhz") if isinstance(clocks, dict) else None
            nominal = {"flop_per_clock_per_sm": round(rate, 1), "sms": sms, "sm_max_mhz": max_mhz,
                       "source": "bwgemm_probe_tensor_rate: tcgen05.mma M=128 N=256 K=16 timed in "
                                 "SM cycles on every SM; peak = SMs x rate x max SM clock"}
            if max_mhz:
                peak = sms * rate * max_mhz * 1e6 / 1e12
                nominal["peak_tflops"] = round(peak, 1)
                nominal["frac"] = round(value / peak, 4)
        except binding.BwgemmError as e:
            nominal = {"unavailable": str(e)}
        roofline["nominal"] = nominal

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(value / PAGES_4096_BF16, 4),
        "vs_baseline_ref": "1772.9 TFLOP/s bf16 4096^3 on B200 (the Blackwell deep dive's "
                           "kernel 8); another machine's number, context only",
        "dtype": shape.dtype,
        "data": "synthetic: seeded N(0,1)/sqrt(K) bf16 A and B, rounded from fp32",
        "config": {"workload": f"{shape.name}: C=A*B^T, M={shape.M} N={shape.N} K={shape.K}, "
                               f"{shape.dtype} in/out, fp32 accumulate",
                   "M": shape.M, "N": shape.N, "K": shape.K,
                   "l2": f"inputs rotate over {len(sets)} copies "
                         f"({len(sets) * shape.algorithmic_bytes / 1e6:.0f} MB > 2x L2)",
                   "parallelism": "single GPU",
                   "kernel_config": kcfg},
        "median_ms": round(median_ms, 5),
        "p10_ms": round(per_sorted[len(per) // 10], 5),
        "p90_ms": round(per_sorted[(9 * len(per)) // 10], 5),
        "per_iteration_note": f"median/p10/p90 over {len(per)} separately event-timed iterations",
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clocks,
        "cublas_tflops": round(shape.flops / cb_s / 1e12, 1),
        "peaks": peaks,
    }
    if shapes:
        # full per-shape records to stderr; the compact summary ends the line
        log(json.dumps({"shapes_detail": shapes}))
    line["shapes"] = {name: compact_shape(rec) for name, rec in shapes.items()}
    print(json.dumps(line, separators=(",", ":")), flush=True)
    plan.close()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=12000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--shape", default=HEADLINE)
    ap.add_argument("--no-extra", action="store_true", help="skip the pages' other shapes")
    ap.add_argument("--fp16-extra", action="store_true",
                    help="also time every other shape in fp16 (adds about a minute)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--idle", type=float, default=2.0,
                    help="idle seconds before the headline's warm-up steps (and cuBLAS's)")
    ap.add_argument("--cooldown", type=float, default=1.0,
                    help="idle seconds before each extra shape (ours and cuBLAS alike)")
    ap.add_argument("--shape-warmup", type=float, default=1.0,
                    help="seconds each extra shape runs before it is timed")
    ap.add_argument("--ref-budget", type=float, default=90.0,
                    help="seconds of oracle work for --impl reference")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.gpus != 1:
        # one GPU only: the GEMM has no multi-GPU path (no sharding, no replicas)
        print(f"bench.py: --gpus {args.gpus} refused: bwgemm runs on one GPU (use --gpus 1)",
              file=sys.stderr, flush=True)
        return 2
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
