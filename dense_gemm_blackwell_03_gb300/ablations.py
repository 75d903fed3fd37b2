"""Ablations of the design steps both pages walk through, on GB300.

``python -m dense_gemm_blackwell_03_gb300.ablations [--shape NAME ...]``
times one launch configuration per row of ``ABLATIONS`` on each named
workload and prints one JSON line per (shape, row): TFLOP/s, GB/s, the
fraction of the roofline ``min(peak, AI x BW)`` and the change against the
default plan.  Each row switches one plan option against the default, so it
measures what that step of the design is worth here:

- CTA pairs (``cta_group::2``, 256-row units) against one CTA per 128-row unit:
  "Matrix Multiplication on NVIDIA's Blackwell", Kernel 5; "Writing a
  Blackwell GEMM by hand", the 2-CTA step.
- Tile width (MMA N 128 / 224 / 256).
- One or two K blocks per TMA copy (a design choice of this library: a copy
  costs the SM's TMA unit about the same time whatever its size).
- Schedules: whole tiles in grouped raster order, stream-K, cluster launch
  control (deep dive Kernel 8), and grouped raster against plain row order
  (deep dive Kernel 9).
- A multicast across two CTA pairs (deep dive Kernel 5's 2x2 cluster; the
  CuTeDSL post's multicast step).
- Split-K: slices in one cluster exchanging through distributed shared
  memory against slices reducing through L2.
- Operand order for small M (C^T = B A^T).
- The whole-K kernels: 64 weight rows per CTA for at most 64 rows of A
  against split-K on 128-row tiles ("Writing a Blackwell GEMM by hand", "Two
  workloads, not one"), and all rows of A on one CTA pair against the main
  kernel for 129 to 256 rows.

Steps fixed at compile time (128B swizzle, the ring depth, the TMEM
double buffer) have no switch in the GEMM.  Two microbenchmarks cover the
measurements the CuTeDSL post makes of them instead:

- ``--load-path``: the load path in isolation, no MMA
  (``bwgemm_bench_load_path``): the GEMM's ring filled by TMA and freed as
  each stage lands, with the 128B swizzle, without it (the same copies,
  plain rows), and in the tensor cores' unswizzled interleaved layout; the
  post's step 4 measured 3.85 TB/s without and 18.5 TB/s with the swizzle on
  B200.
- ``--epilogue-share``: the epilogue's share of an unmodified launch, from
  the kernel's own per-unit timestamps (the post's step 5: at most 13 of
  109 us at 4096^3 on B200).

``python -m dense_gemm_blackwell_03_gb300.ablations --table FILE`` turns the
JSON lines of an earlier run (FILE) into the markdown table of the timed
rows, without a GPU.  Timing: each row runs
about ``--warmup`` seconds, then the median of three blocks of about 0.1 s
is taken, with CUDA events on the launching stream; inputs rotate over
copies larger than L2.
"""
from __future__ import annotations

import argparse
import json
import statistics
import time

# (label, plan options, what the row isolates)
ABLATIONS = [
    ("default", {}, "the planner's choice"),
    ("one CTA per unit", {"variant": 1}, "CTA pairs (cta_group::2) off"),
    ("CTA pair", {"variant": 2}, "CTA pairs forced"),
    ("tile N 128", {"tile_n": 128}, "narrower MMA N"),
    ("tile N 224", {"tile_n": 224, "variant": 2, "swap_ab": 1}, "224-column pair tiles"),
    ("tile N 256", {"tile_n": 256}, "256-column tiles"),
    ("1 K block per copy", {"copy_kblocks": 1}, "one TMA copy per K block and operand"),
    ("2 K blocks per copy", {"copy_kblocks": 2}, "one TMA copy per two K blocks"),
    ("whole tiles", {"schedule": 1}, "static persistent schedule, no stream-K"),
    ("stream-K", {"schedule": 2}, "stream-K over the last wave"),
    ("cluster launch control", {"schedule": 3}, "clusters cancel pending launches"),
    ("raster group 1", {"raster_group": 1}, "row-order tiles instead of groups of 8"),
    ("A multicast", {"multicast": 2}, "two pairs share each A tile"),
    ("split-K through L2", {"cluster_split": 1}, "clustered split-K exchange off"),
    ("operands in order", {"swap_ab": 1}, "C^T = B A^T off"),
    ("whole-K kernel off", {"skinny": 1}, "split-K on 128-row tiles instead of 64 weight rows per CTA, whole K"),
    ("whole-K pair kernel", {"wholek": 2}, "all rows of A on one CTA pair, narrow weight blocks, whole K"),
    ("whole-K pair kernel off", {"wholek": 1}, "the main kernel instead of the whole-K pair kernel"),
]

DEFAULT_SHAPES = ["square4096", "prefill_attn_out", "decode_attn_out", "decode_qkv", "tail_m64"]

SHAPE_LABELS = {"square4096": "4096^3", "prefill_attn_out": "prefill 8192^3",
                "decode_attn_out": "decode M=256 N=K=8192", "decode_qkv": "decode M=256 N=10240 K=8192",
                "tail_m64": "tail M=64 N=K=8192"}


def describe(cfg: dict) -> str:
    """Short description of a launch configuration (the default rows' label)."""
    if cfg.get("skinny"):
        form = "CTA pairs (M = 128)" if cfg.get("variant") == 2 else "1 CTA (M = 64)"
        return f"whole-K, 64 weight rows per CTA, {form}, N = {cfg.get('tile_n')}"
    if cfg.get("wholek"):
        return f"whole-K pairs, all rows of A, {cfg.get('tile_n')} weight rows per pair"
    parts = ["swapped" if cfg.get("swap_ab") == 1 else None,
             "pairs" if cfg.get("variant") == 2 else "1 CTA",
             str(cfg.get("tile_n")),
             f"{cfg.get('copy_kblocks')} K blocks/copy" if cfg.get("copy_kblocks") == 2 else None]
    if cfg.get("split_k", 1) > 1:
        where = "in clusters" if cfg.get("cluster_split") == 1 else "through L2"
        parts.append(f"split-K {cfg['split_k']} {where}")
    else:
        parts.append({1: "whole tiles", 2: "stream-K", 3: "cluster launch control"}.get(cfg.get("schedule"),
                                                                                       "schedule ?"))
    return ", ".join(p for p in parts if p)


def markdown_table(rows) -> str:
    """The timed rows of a run as a markdown table (untimed rows are left out)."""
    out = ["| shape | row | us | TFLOP/s | fraction | vs default |", "|---|---|---:|---:|---:|---:|"]
    for r in rows:
        if "us" not in r:
            continue
        label = r["row"]
        if label == "default":
            label = f"default ({describe(r.get('config', {}))})"
        vs = r.get("vs_default")
        out.append(f"| {SHAPE_LABELS.get(r['shape'], r['shape'])} | {label} | {r['us']:.2f} | "
                   f"{r['tflops']:.1f} | {r['roofline_frac']:.3f} | {'1' if vs is None else f'{vs:.3f}'} |")
    return "\n".join(out)


# the CuTeDSL post's figures (B200), quoted beside the GB300 rows
PAGE_LOAD_PATH_TBS = {0: 18.5, 1: 3.85}
LOAD_PATH_STAGES = 6
LOAD_PATH_KBLOCKS = 4096
EPILOGUE_SHAPES = ["square4096", "prefill_attn_out", "decode_attn_out", "decode_qkv", "tail_m64"]


def load_path_table(rows) -> str:
    """Markdown table of --load-path rows."""
    out = ["| layout | copies per 32 KiB stage | TB/s (GB300) | vs 128B swizzle | post, B200 (TB/s) |",
           "|---|---:|---:|---:|---:|"]
    for r in rows:
        page = PAGE_LOAD_PATH_TBS.get(r["layout"])
        out.append(f"| {r['row']} | {r['copies_per_stage']} | {r['gbs'] / 1e3:.2f} | "
                   f"{r['vs_swizzle']:.3f} | {'' if page is None else page} |")
    return "\n".join(out)


def epilogue_table(rows) -> str:
    """Markdown table of --epilogue-share rows."""
    out = ["| shape | span (us) | units per CTA | epilogue busy per CTA (us) | busy share | "
           "exposed after last MMA (us) | exposed share |",
           "|---|---:|---:|---:|---:|---:|---:|"]
    for r in rows:
        e = r["epilogue"]
        out.append(f"| {SHAPE_LABELS.get(r['shape'], r['shape'])} | {e['span_us']:.2f} | "
                   f"{r['units_per_cta']:.2f} | {e['busy_us_per_cta']:.2f} | {e['busy_share']:.3f} | "
                   f"{e['exposed_us']:.2f} | {e['exposed_share']:.3f} |")
    return "\n".join(out)


def run_load_path(device: int = 0):
    """The three layouts of bwgemm_bench_load_path, as JSON rows."""
    from . import binding
    rows = []
    for layout in (0, 1, 2):
        gbs, ms = binding.bench_load_path(layout, 0, 0, LOAD_PATH_STAGES, LOAD_PATH_KBLOCKS, device)
        rows.append({"kind": "load_path", "layout": layout, "row": binding.LOAD_PATH_LAYOUTS[layout],
                     "copies_per_stage": 16 if layout == 2 else 2, "stages": LOAD_PATH_STAGES,
                     "kblocks_per_cta": LOAD_PATH_KBLOCKS, "gbs": round(gbs, 1), "ms": round(ms, 4)})
    for r in rows:
        r["vs_swizzle"] = round(r["gbs"] / rows[0]["gbs"], 4)
    return rows


def run_epilogue_share(names, warmup: int = 6):
    """One traced launch of each named shape (default plan, after warm-up
    launches on rotating inputs): the epilogue's share, as JSON rows."""
    import torch

    from . import binding, timeline
    from .workloads import SHAPES, make_inputs
    rows = []
    for name in names:
        s = SHAPES[name]
        sets = [make_inputs(s, device="cuda", seed=100 + i) for i in range(3)]
        with binding.Plan(0, trace=1) as plan:
            for i in range(warmup):
                plan.gemm(*sets[i % 3])
            torch.cuda.synchronize()
            plan.gemm(*sets[0])
            if plan.status() != 0:
                raise SystemExit(f"device status error on {name}")
            trace = plan.read_trace()
            cfg = plan.last_config()
        per = timeline.units(trace)
        rows.append({"kind": "epilogue_share", "shape": name, "epilogue": timeline.epilogue_share(trace),
                     "units_per_cta": round(sum(len(u) for u in per) / max(1, len(per)), 3),
                     "config": {k: cfg[k] for k in ("variant", "tile_n", "split_k", "schedule", "grid")}})
        del sets
        torch.cuda.empty_cache()
    return rows


def _steady(run, sets, warmup_s):
    """Seconds per launch in steady state (CUDA events, median of 3 blocks)."""
    import torch
    stream = torch.cuda.current_stream()

    def block(n):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            run(*sets[i % len(sets)])
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3

    pilot = block(10) / 10
    n = int(min(5000, max(20, 0.1 / max(pilot, 1e-7))))
    t_end = time.perf_counter() + warmup_s
    while time.perf_counter() < t_end:
        block(n)
    return statistics.median(block(n) / n for _ in range(3))


def _peaks():
    import os
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def _input_sets(shape, l2_bytes):
    import math

    import torch

    from .workloads import TORCH_DTYPES, make_inputs
    n = 1 if shape.algorithmic_bytes >= 2 * l2_bytes else min(3, math.ceil(3 * l2_bytes / shape.algorithmic_bytes))
    sets = []
    for i in range(n):
        A, B = make_inputs(shape, device="cuda", seed=None if i == 0 else 7919 * i + 17)
        C = torch.empty((shape.M, shape.N), dtype=TORCH_DTYPES[shape.dtype], device="cuda")
        sets.append((A, B, C))
    return sets


def main(argv=None) -> int:
    import torch

    from . import binding
    from .workloads import SHAPES

    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--shape", action="append", choices=sorted(SHAPES),
                    help="workload (repeatable; default: 4096^3, prefill attention-out, "
                         "decode attention-out, M = 64 tail)")
    ap.add_argument("--warmup", type=float, default=0.3, help="seconds of each row's own load before timing")
    ap.add_argument("--cooldown", type=float, default=0.5, help="idle seconds before each row")
    ap.add_argument("--table", metavar="FILE",
                    help="print the markdown table of an earlier run's JSON lines and exit (no GPU)")
    ap.add_argument("--load-path", action="store_true",
                    help="also run the load-path microbenchmark (no MMA; three layouts)")
    ap.add_argument("--epilogue-share", action="store_true",
                    help="also measure the epilogue's share of one traced launch per shape")
    ap.add_argument("--only-microbench", action="store_true",
                    help="run only the microbenchmarks asked for, not the plan-option rows")
    args = ap.parse_args(argv)
    if args.table:
        with open(args.table) as f:
            rows = [json.loads(line) for line in f if line.startswith("{")]
        gemm_rows = [r for r in rows if r.get("kind") is None]
        if gemm_rows:
            print(markdown_table(gemm_rows))
        lp = [r for r in rows if r.get("kind") == "load_path"]
        if lp:
            print("\n" + load_path_table(lp))
        ep = [r for r in rows if r.get("kind") == "epilogue_share"]
        if ep:
            print("\n" + epilogue_table(ep))
        return 0
    binding.load_library(build_if_missing=True)
    if args.load_path:
        for row in run_load_path():
            print(json.dumps(row), flush=True)
    if args.epilogue_share:
        for row in run_epilogue_share(args.shape or EPILOGUE_SHAPES):
            print(json.dumps(row), flush=True)
    if args.only_microbench:
        return 0
    hbm_gbs, tflops_peak, peak_src = _peaks()
    props = torch.cuda.get_device_properties(0)
    l2_bytes = int(getattr(props, "L2_cache_size", 129 * 10 ** 6)) or 129 * 10 ** 6
    for name in args.shape or DEFAULT_SHAPES:
        s = SHAPES[name]
        sets = _input_sets(s, l2_bytes)
        ai = s.flops / s.algorithmic_bytes
        attainable = min(tflops_peak, ai * hbm_gbs / 1e3)
        base_t = None
        base_cfg = None
        for label, opts, what in ABLATIONS:
            row = {"shape": name, "row": label, "options": opts, "isolates": what}
            try:
                plan = binding.Plan(0, **opts)
                plan.gemm(*sets[0][:2], out=sets[0][2])
            except binding.BwgemmError as e:
                row["result"] = f"not applicable: {e}"
                print(json.dumps(row), flush=True)
                continue
            cfg = plan.last_config()
            if base_cfg is not None and cfg == base_cfg:
                row["result"] = "same configuration as the default"
                print(json.dumps(row), flush=True)
                plan.close()
                continue
            torch.cuda.synchronize()
            time.sleep(args.cooldown)
            t = _steady(lambda A, B, C: plan.gemm(A, B, out=C), sets, args.warmup)
            status = plan.status()
            plan.close()
            if status != 0:
                raise SystemExit(f"device status {status} on {name} / {label}")
            tflops = s.flops / t / 1e12
            row.update({"us": round(t * 1e6, 2), "tflops": round(tflops, 1),
                        "gbs": round(s.algorithmic_bytes / t / 1e9, 1),
                        "roofline_frac": round(tflops / attainable, 4), "peak_source": peak_src,
                        "config": {k: cfg[k] for k in ("variant", "tile_n", "split_k", "schedule", "grid",
                                                       "copy_kblocks", "multicast", "cluster_split",
                                                       "swap_ab", "raster_group", "skinny", "wholek")}})
            if base_t is None:
                base_t, base_cfg = t, cfg
            else:
                row["vs_default"] = round(base_t / t, 4)
            print(json.dumps(row), flush=True)
        del sets
        torch.cuda.empty_cache()
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
