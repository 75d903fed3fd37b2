"""Host-side checks of the ablation table (no GPU): every row names real plan
options, and on each default workload it either plans or is refused with a
library status (never a Python error)."""
from __future__ import annotations

import pytest

from dense_gemm_blackwell_03_gb300 import ablations, binding
from dense_gemm_blackwell_03_gb300.workloads import SHAPES


def test_rows_are_plan_options():
    labels = [label for label, _, _ in ablations.ABLATIONS]
    assert labels[0] == "default" and len(set(labels)) == len(labels)
    for _, opts, what in ablations.ABLATIONS:
        binding.make_options(**opts)  # raises TypeError on an unknown option
        assert what


@pytest.mark.parametrize("name", ablations.DEFAULT_SHAPES)
def test_rows_plan_or_are_refused(name):
    s = SHAPES[name]
    planned = 0
    for _, opts, _ in ablations.ABLATIONS:
        try:
            binding.select_config(152, s.M, s.N, s.K, max_pairs=76, max_quads=36, **opts)
            planned += 1
        except binding.BwgemmError as e:
            assert e.status in (1, 3)  # invalid argument / unsupported for this shape
    assert planned >= len(ablations.ABLATIONS) - 3


def test_markdown_table_from_rows():
    rows = [
        {"shape": "decode_attn_out", "row": "default", "us": 32.17, "tflops": 1068.0, "roofline_frac": 0.654,
         "config": {"variant": 2, "tile_n": 256, "split_k": 2, "schedule": 1, "copy_kblocks": 1,
                    "cluster_split": 1, "swap_ab": 0}},
        {"shape": "decode_attn_out", "row": "CTA pair", "result": "same configuration as the default"},
        {"shape": "decode_attn_out", "row": "one CTA per unit", "us": 40.34, "tflops": 851.9,
         "roofline_frac": 0.522, "vs_default": 0.7976},
        {"shape": "tail_m64", "row": "default", "us": 27.01, "tflops": 318.0, "roofline_frac": 0.745,
         "config": {"variant": 1, "tile_n": 64, "split_k": 2, "schedule": 1, "copy_kblocks": 1,
                    "cluster_split": 1, "swap_ab": 1}},
    ]
    lines = ablations.markdown_table(rows).splitlines()
    assert lines[0].startswith("| shape | row |") and len(lines) == 2 + 3  # untimed rows left out
    assert lines[2] == ("| decode M=256 N=K=8192 | default (pairs, 256, split-K 2 in clusters) | 32.17 | "
                        "1068.0 | 0.654 | 1 |")
    assert lines[3].endswith("| 40.34 | 851.9 | 0.522 | 0.798 |")
    assert "default (swapped, 1 CTA, 64, split-K 2 in clusters)" in lines[4]


def test_load_path_and_epilogue_tables():
    lp = [{"kind": "load_path", "layout": 0, "row": "128B swizzle", "copies_per_stage": 2, "gbs": 20000.0,
           "vs_swizzle": 1.0},
          {"kind": "load_path", "layout": 1, "row": "no swizzle, plain rows (same copies)",
           "copies_per_stage": 2, "gbs": 5000.0, "vs_swizzle": 0.25}]
    lines = ablations.load_path_table(lp).splitlines()
    assert len(lines) == 4
    assert lines[2] == "| 128B swizzle | 2 | 20.00 | 1.000 | 18.5 |"
    assert lines[3].endswith("| 5.00 | 0.250 | 3.85 |")
    ep = [{"kind": "epilogue_share", "shape": "square4096", "units_per_cta": 2.5,
           "epilogue": {"span_us": 84.0, "busy_us_per_cta": 9.0, "busy_share": 0.1071,
                        "exposed_us": 3.0, "exposed_share": 0.0357}}]
    lines = ablations.epilogue_table(ep).splitlines()
    assert lines[2] == "| 4096^3 | 84.00 | 2.50 | 9.00 | 0.107 | 3.00 | 0.036 |"


def test_epilogue_share_from_stamps():
    import numpy as np

    from dense_gemm_blackwell_03_gb300 import timeline
    from dense_gemm_blackwell_03_gb300.binding import (TRACE_ENTRY, TRACE_EXIT, TRACE_UNIT0,
                                                       TRACE_UNITS)
    tr = np.zeros((2, TRACE_UNIT0 + 4 * TRACE_UNITS), dtype=np.uint64)
    # CTA 0: two units; MMAs 1000-5000 and 5000-9000 ns, epilogues 5100-6100 and 9100-10100
    tr[0, TRACE_ENTRY], tr[0, TRACE_EXIT] = 1000, 10500
    tr[0, TRACE_UNIT0:TRACE_UNIT0 + 8] = [1000, 5000, 5100, 6100, 5000, 9000, 9100, 10100]
    # CTA 1: one unit, epilogue 500 ns after its last commit
    tr[1, TRACE_ENTRY], tr[1, TRACE_EXIT] = 1000, 11000
    tr[1, TRACE_UNIT0:TRACE_UNIT0 + 4] = [1200, 9500, 9600, 10000]
    e = timeline.epilogue_share(tr)
    assert e["ctas"] == 2 and e["span_us"] == 10.0
    assert e["busy_us_per_cta"] == round((2000 + 400) / 2 / 1e3, 3)
    assert e["exposed_us"] == round((1100 + 500) / 2 / 1e3, 3)
    assert e["exposed_share"] == round(800 / 10000, 4)
