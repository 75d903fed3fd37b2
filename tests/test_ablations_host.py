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
