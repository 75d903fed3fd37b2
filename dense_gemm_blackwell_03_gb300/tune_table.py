"""Offline sweep behind the library's table of tuned options.

"Matrix Multiplication on NVIDIA's Blackwell" (experimental results, the
Gemma-3-27B shape) picks the MMA shape, pipeline depth and swizzle per
problem shape with an autotuner.  Here the planner's rules choose a launch
configuration from the shape alone; this sweep checks them on the pages'
shapes:

    python -m dense_gemm_blackwell_03_gb300.tune_table --sweep > sweep.jsonl   # GB300
    python -m dense_gemm_blackwell_03_gb300.tune_table --table sweep.jsonl     # markdown, no GPU
    python -m dense_gemm_blackwell_03_gb300.tune_table --header sweep.jsonl    # csrc/tuned_table.h, no GPU

For each shape ``--sweep`` runs ``bwgemm_tune`` (every candidate of its fixed
list timed back to back with CUDA events, the table off), then times the
rules' choice and the tuned choice again in steady state, in alternating
order (``ROUNDS`` rounds of: idle, warm-up, median of three ~0.1 s blocks),
and prints one JSON line.  ``--header`` keeps the shapes whose tuned choice
was at least ``MIN_GAIN`` faster and writes them as the table that
``select_config`` applies (after a rebuild).  The table is keyed by (M, N, K):
bf16 and fp16 run the same instructions, so the bf16 sweep stands for both.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import time

HERE = os.path.dirname(os.path.abspath(__file__))
HEADER_PATH = os.path.join(HERE, "csrc", "tuned_table.h")

# the pages' shapes (one per (M, N, K); the fp16 square shares the bf16 entry)
SWEEP_SHAPES = ["square4096", "prefill_attn_out", "prefill_mlp_up", "decode_attn_out", "decode_qkv",
                "decode_mlp_up", "decode_mlp_down", "gemma_512x8192x5376", "tail_m1", "tail_m16",
                "tail_m64", "tail_m200"]
# the plan options a table entry may set, in the order of TunedEntry
OPTION_KEYS = ("variant", "tile_n", "split_k", "schedule", "copy_kblocks", "cluster_split", "raster_group",
               "swap_ab", "multicast", "skinny")
CONFIG_KEYS = ("variant", "tile_n", "split_k", "schedule", "copy_kblocks", "cluster_split", "raster_group",
               "swap_ab", "multicast", "grid", "stages", "skinny", "wholek")
MIN_GAIN = 1.015  # tuned time at least 1.5 % below the rules' time
ROUNDS = 3


def options_of(cfg: dict) -> dict:
    """Plan options that reproduce a launch configuration exactly."""
    if cfg.get("skinny"):
        return {k: 0 for k in OPTION_KEYS if k != "skinny"} | {"skinny": 2}
    if cfg.get("wholek"):  # the whole-K pair kernel: its own planner rule, no table entry
        return {k: 0 for k in OPTION_KEYS}
    return {
        "variant": int(cfg["variant"]),
        "tile_n": int(cfg["tile_n"]),
        "split_k": int(cfg["split_k"]),
        "schedule": int(cfg["schedule"]),
        "copy_kblocks": int(cfg["copy_kblocks"]),
        "cluster_split": 2 if cfg["cluster_split"] else 1,
        "raster_group": int(cfg["raster_group"]),
        "swap_ab": 2 if cfg["swap_ab"] else 1,
        "multicast": 2 if cfg["multicast"] == 2 else 1,
        "skinny": 1,
    }


def same_config(a: dict, b: dict) -> bool:
    return all(a[k] == b[k] for k in CONFIG_KEYS)


def header_text(rows, min_gain: float = MIN_GAIN) -> str:
    """C++ source of tuned_table.h from sweep rows (those gaining >= min_gain)."""
    keep = [r for r in rows if r.get("options") and r.get("gain", 0.0) >= min_gain]
    lines = [
        "// tuned_table.h -- written by `python -m dense_gemm_blackwell_03_gb300.tune_table",
        "// --header`: plan options that the offline sweep over the pages' shapes measured",
        "// faster than the planner's own choice (steady-state CUDA-event timing on",
        "// GB300, alternating order).  select_config applies an entry when the shape",
        "// matches exactly and the caller left every option it sets on automatic.",
        "#pragma once",
        "",
        "#include <cstdint>",
        "",
        "namespace bwgemm {",
        "",
        "struct TunedEntry {",
        "    int64_t M, N, K;",
        "    // the options the entry sets (0 = automatic, as in bwgemm_plan_options_t)",
        "    int32_t variant, tile_n, split_k, schedule, copy_kblocks, cluster_split, raster_group, swap_ab,",
        "        multicast, skinny;",
        "};",
        "",
        "// the last entry (M = 0) ends the table",
        "constexpr TunedEntry kTunedTable[] = {",
    ]
    for r in keep:
        o = r["options"]
        vals = ", ".join(str(int(o[k])) for k in OPTION_KEYS)
        lines.append(f"    {{{r['M']}, {r['N']}, {r['K']}, {vals}}},  // {r['shape']}: "
                     f"{r['rules_us']:.2f} -> {r['tuned_us']:.2f} us")
    lines += ["    {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0},", "};", "", "}  // namespace bwgemm", ""]
    return "\n".join(lines)


def markdown(rows) -> str:
    out = ["| shape | rules' choice | us | tuned choice | us | tuned / rules | in table |",
           "|---|---|---:|---|---:|---:|:---:|"]
    for r in rows:
        def d(c):
            if c.get("skinny"):
                return f"whole-K, 64 weight rows per CTA ({c['variant']}sm), N {c['tile_n']}"
            if c.get("wholek"):
                return f"whole-K pairs, {c['tile_n']} weight rows per pair"
            mc = "x2 multicast" if c.get("multicast") == 2 else ""
            sk = f"split {c['split_k']}" + (" in clusters" if c.get("cluster_split") else "") \
                if c.get("split_k", 1) > 1 else {1: "tiles", 2: "stream-K", 3: "CLC"}.get(c.get("schedule"), "?")
            sw = "swapped " if c.get("swap_ab") else ""
            return f"{sw}{c['variant']}sm {c['tile_n']}, {sk}, {c['copy_kblocks']} kb/copy, G{c['raster_group']} {mc}".strip()
        same = r.get("same")
        out.append(f"| {r['shape']} | {d(r['rules'])} | {r['rules_us']:.2f} | "
                   f"{'(same)' if same else d(r['tuned'])} | {r['tuned_us']:.2f} | "
                   f"{r['tuned_us'] / r['rules_us']:.3f} | {'yes' if r.get('gain', 0) >= MIN_GAIN else ''} |")
    return "\n".join(out)


def _steady(plan, sets, warmup_s):
    from .ablations import _steady as steady
    return steady(lambda A, B, C: plan.gemm(A, B, out=C), sets, warmup_s)


def sweep(names, iters_short=200, iters_long=30, warmup_s=0.4, cooldown_s=0.6):
    import torch

    from . import binding
    from .ablations import _input_sets
    from .workloads import SHAPES
    binding.load_library(build_if_missing=True)
    for name in names:
        s = SHAPES[name]
        sets = _input_sets(s, 129 * 10 ** 6)
        A, B, C = sets[0]
        rules = binding.Plan(0, tuned_table=1)
        rules.gemm(A, B, out=C)
        cfg_rules = rules.last_config()
        tuner = binding.Plan(0, tuned_table=1)
        iters = iters_short if s.flops < 2e11 else iters_long
        cfg_tuned = tuner.tune(A, B, out=C, iters=iters)
        assert tuner.status() == 0
        tuner.close()
        opts = options_of(cfg_tuned)
        row = {"shape": name, "M": s.M, "N": s.N, "K": s.K,
               "rules": {k: cfg_rules[k] for k in CONFIG_KEYS},
               "tuned": {k: cfg_tuned[k] for k in CONFIG_KEYS}}
        same = same_config(cfg_rules, cfg_tuned)
        cand = binding.Plan(0, tuned_table=1, **opts)
        cand.gemm(A, B, out=C)
        assert same_config(cand.last_config(), cfg_tuned), "options do not reproduce the tuned configuration"
        # the same configuration is timed once per round; different ones alternate
        timed = ((rules, []),) if same else ((rules, []), (cand, []))
        for _ in range(ROUNDS):
            for plan, acc in timed:
                torch.cuda.synchronize()
                time.sleep(cooldown_s)
                acc.append(_steady(plan, sets, warmup_s))
        assert rules.status() == 0 and cand.status() == 0
        t_rules = timed[0][1]
        t_tuned = timed[-1][1]
        tr = statistics.median(t_rules)
        tt = statistics.median(t_tuned)
        row.update({"same": same, "rules_us": round(tr * 1e6, 2), "tuned_us": round(tt * 1e6, 2),
                    "gain": round(tr / tt, 4), "options": None if same else opts,
                    "rounds_us": {"rules": [round(x * 1e6, 2) for x in t_rules],
                                  "tuned": [round(x * 1e6, 2) for x in t_tuned]}})
        print(json.dumps(row), flush=True)
        rules.close()
        cand.close()
        del sets, A, B, C
        torch.cuda.empty_cache()


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--sweep", action="store_true", help="run the sweep on cuda:0, JSON lines to stdout")
    ap.add_argument("--shape", action="append", help="sweep only these shapes (repeatable)")
    ap.add_argument("--table", metavar="FILE", help="markdown table of a sweep's JSON lines (no GPU)")
    ap.add_argument("--header", metavar="FILE", help="write csrc/tuned_table.h from a sweep's JSON lines")
    ap.add_argument("--out", default=HEADER_PATH, help="where --header writes")
    args = ap.parse_args(argv)
    if args.table or args.header:
        with open(args.table or args.header) as f:
            rows = [json.loads(line) for line in f if line.startswith("{")]
        if args.table:
            print(markdown(rows))
        else:
            with open(args.out, "w") as f:
                f.write(header_text(rows))
            print(f"wrote {args.out}")
        return 0
    if args.sweep:
        sweep(args.shape or SWEEP_SHAPES)
        return 0
    ap.print_help()
    return 2


if __name__ == "__main__":
    raise SystemExit(main())
