"""Summaries of a launch timeline read with ``Plan.read_trace()``.

The kernel stamps ``%globaltimer`` (ns) at fixed points of each CTA's life
(entry, prologue done, first/last TMA load, epilogue done, exit) and, per work
unit, when the MMA warp starts and commits it and when the epilogue starts
and finishes it.  ``summarize`` turns the raw (ctas x slots) array into the
phase durations that explain a kernel's time: launch skew, prologue, pipeline
fill, MMA issue time per CTA, epilogue time per unit and the exit tail.
"""
from __future__ import annotations

import numpy as np

from .binding import (TRACE_ENTRY, TRACE_EPI_DONE, TRACE_EXIT, TRACE_FIRST_LOAD,
                      TRACE_LAST_LOAD, TRACE_READY, TRACE_UNIT0, TRACE_UNITS)


def _stat(x) -> dict:
    x = np.asarray([v for v in x if v is not None], dtype=np.float64)
    if x.size == 0:
        return {"n": 0}
    return {"n": int(x.size), "min": round(float(x.min()), 3), "mean": round(float(x.mean()), 3),
            "max": round(float(x.max()), 3)}


def units(trace: np.ndarray):
    """Per CTA, the list of (mma_start, mma_end, epi_start, epi_end) in ns
    (entries 0 when that role did not stamp it)."""
    out = []
    for row in trace:
        u = []
        for k in range(TRACE_UNITS):
            s = row[TRACE_UNIT0 + 4 * k: TRACE_UNIT0 + 4 * k + 4]
            if not s.any():
                break
            u.append(tuple(int(v) for v in s))
        out.append(u)
    return out


def epilogue_share(trace: np.ndarray) -> dict:
    """How much of a launch the epilogue takes ("Writing a Blackwell GEMM by
    hand", step 5: measure a stage's share of the kernel before optimising
    it), from the stamps of an unmodified launch:

    - busy: the epilogue warps' time with an accumulator in hand (from seeing
      it ready to the unit's last store issued), summed over a CTA's units,
      as a share of the launch's span; the TMEM double buffer overlaps most of
      it with the next unit's MMAs;
    - exposed: per CTA, the time from its last MMA commit to the end of its
      last epilogue, which nothing overlaps; as microseconds and as a share
      of the span.
    """
    tr = np.asarray(trace, dtype=np.int64)
    tr = tr[tr[:, TRACE_ENTRY] > 0]
    if tr.shape[0] == 0:
        return {"ctas": 0}
    span = float(tr[:, TRACE_EXIT].max() - tr[:, TRACE_ENTRY].min())
    busy, exposed = [], []
    for ulist in units(tr):
        done = [u for u in ulist if u[2] > 0 and u[3] > 0]
        if not done:
            continue
        busy.append(sum(u[3] - u[2] for u in done))
        last_commit = max((u[1] for u in ulist if u[1] > 0), default=0)
        if last_commit:
            exposed.append(max(0, max(u[3] for u in done) - last_commit))
    if not busy or span <= 0:
        return {"ctas": int(tr.shape[0])}
    return {"ctas": int(tr.shape[0]), "span_us": round(span / 1e3, 3),
            "busy_us_per_cta": round(float(np.mean(busy)) / 1e3, 3),
            "busy_share": round(float(np.mean(busy)) / span, 4),
            "exposed_us": round(float(np.mean(exposed)) / 1e3, 3) if exposed else None,
            "exposed_share": round(float(np.mean(exposed)) / span, 4) if exposed else None}


def summarize(trace: np.ndarray) -> dict:
    """Phase durations in microseconds over all CTAs of one launch."""
    tr = np.asarray(trace, dtype=np.int64)
    entry = tr[:, TRACE_ENTRY]
    live = entry > 0
    tr = tr[live]
    if tr.shape[0] == 0:
        return {"ctas": 0}
    t0 = int(tr[:, TRACE_ENTRY].min())
    us = lambda a, b: (int(b) - int(a)) / 1e3 if a > 0 and b > 0 else None  # noqa: E731
    per_unit = units(tr)
    mma_busy, epi_len, first_mma_wait, tails, unit_gaps = [], [], [], [], []
    for row, ulist in zip(tr, per_unit):
        starts = [u[0] for u in ulist if u[0] > 0]
        if starts:
            first_mma_wait.append(us(row[TRACE_READY], starts[0]))
            mma_busy.append(sum(us(u[0], u[1]) or 0.0 for u in ulist if u[0] > 0 and u[1] > 0))
        for u in ulist:
            if u[2] > 0 and u[3] > 0:
                epi_len.append(us(u[2], u[3]))
            if u[1] > 0 and u[2] > 0:
                unit_gaps.append(us(u[1], u[2]))  # MMA commit -> epilogue sees the accumulator
        ends = [u[3] for u in ulist if u[3] > 0]
        if ends and row[TRACE_EXIT] > 0:
            tails.append(us(max(ends), row[TRACE_EXIT]))
    return {
        "ctas": int(tr.shape[0]),
        "span_us": round((int(tr[:, TRACE_EXIT].max()) - t0) / 1e3, 3),
        "entry_skew_us": _stat((tr[:, TRACE_ENTRY] - t0) / 1e3),
        "prologue_us": _stat([us(a, b) for a, b in zip(tr[:, TRACE_ENTRY], tr[:, TRACE_READY])]),
        "first_load_after_entry_us": _stat([us(a, b) for a, b in
                                            zip(tr[:, TRACE_ENTRY], tr[:, TRACE_FIRST_LOAD])]),
        "first_mma_after_ready_us": _stat(first_mma_wait),
        "mma_issue_us_per_cta": _stat(mma_busy),
        "commit_to_epilogue_us": _stat(unit_gaps),
        "epilogue_per_unit_us": _stat(epi_len),
        "last_load_us": _stat((tr[:, TRACE_LAST_LOAD][tr[:, TRACE_LAST_LOAD] > 0] - t0) / 1e3),
        "epilogue_done_us": _stat((tr[:, TRACE_EPI_DONE][tr[:, TRACE_EPI_DONE] > 0] - t0) / 1e3),
        "exit_us": _stat((tr[:, TRACE_EXIT] - t0) / 1e3),
        "tail_after_last_epilogue_us": _stat(tails),
        "units_per_cta": _stat([len(u) for u in per_unit]),
    }


def main(argv=None) -> int:
    """``python -m dense_gemm_blackwell_03_gb300.timeline --shape NAME``: trace
    one launch of a named workload (after warm-up launches on rotating input
    copies) and print its phase summary as JSON."""
    import argparse
    import json

    import torch

    from . import binding
    from .workloads import SHAPES, make_inputs

    ap = argparse.ArgumentParser(description=main.__doc__)
    ap.add_argument("--shape", default="decode_attn_out", choices=sorted(SHAPES))
    ap.add_argument("--schedule", type=int, default=0)
    ap.add_argument("--split-k", type=int, default=0)
    ap.add_argument("--warmup", type=int, default=6)
    ap.add_argument("--opt", action="append", default=[], metavar="NAME=INT",
                    help="any other plan option (repeatable), e.g. --opt multicast=2")
    args = ap.parse_args(argv)
    opts = {}
    for kv in args.opt:
        name, _, value = kv.partition("=")
        opts[name] = int(value)
    s = SHAPES[args.shape]
    sets = [make_inputs(s, device="cuda", seed=100 + i) for i in range(3)]
    with binding.Plan(0, trace=1, schedule=args.schedule, split_k=args.split_k, **opts) as plan:
        for i in range(args.warmup):
            plan.gemm(*sets[i % 3])
        torch.cuda.synchronize()
        plan.gemm(*sets[0])
        if plan.status() != 0:
            raise SystemExit("device status error")
        trace = plan.read_trace()
        cfg = plan.last_config()
    spans = [(u[1] - u[0]) / 1e3 for row in units(trace) for u in row if u[0] and u[1]]
    out = {"shape": args.shape, "config": cfg, "summary": summarize(trace),
           "mma_span_us_per_unit": _stat(spans), "epilogue": epilogue_share(trace)}
    print(json.dumps(out))
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
