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
