"""The allocation-free split-K entry point against the plan-based one.

bwgemm_run_splitk_noalloc serves callers that cannot call cudaMalloc (a
memory manager that already reserved the device, a fixed device footprint,
loops that must not risk the synchronisation cudaMalloc / cudaFree can
cause): its split-K scratch lives in a fixed array inside the library.  Here
it must give the same C as bwgemm_run with the same split, on two calls in a
row (the second call finds the first call's leftovers in the shared array),
and refuse shapes whose scratch does not fit the array.

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

from dense_gemm_blackwell_03_gb300 import binding
from dense_gemm_blackwell_03_gb300.workloads import bits_of, make_matrix
from parity import compare

pytestmark = pytest.mark.gpu

WORKSPACE = 7


def run_noalloc(lib, A, B, C, split):
    M, K = A.shape
    N = B.shape[0]
    stream = ctypes.c_void_p(int(torch.cuda.current_stream().cuda_stream))
    return lib.bwgemm_run_splitk_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                         A.stride(0), B.stride(0), C.stride(0), binding.BF16,
                                         split, stream)


@pytest.mark.parametrize("M,N,K,dist,split", [
    (256, 512, 1600, "int2", 3),     # CTA-pair tiles, exact integers
    (100, 384, 4096, "normal", 4),   # single-CTA tiles, ragged M, N(0,1) inputs
    (300, 264, 1000, "normal", 2),   # ragged M, N and K
])
def test_noalloc_matches_plan_entry_point(M, N, K, dist, split):
    assert torch.cuda.is_available()
    lib = binding.load_library(build_if_missing=True)
    A = make_matrix(M, K, dist, seed=1200 + split, device="cuda")
    B = make_matrix(N, K, dist, seed=1300 + split, device="cuda")
    with binding.Plan(0, split_k=split) as plan:
        want = plan.gemm(A, B)
        assert plan.status() == 0
        assert plan.last_config()["split_k"] == split
    ref = bits_of(want)
    for _ in range(2):  # two calls in a row share (and reuse) the fixed scratch
        C = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
        assert run_noalloc(lib, A, B, C, split) == 0
        torch.cuda.synchronize()
        compare(bits_of(C), ref, "bf16", K, exact=(dist == "int2"))


def test_noalloc_refuses_scratch_beyond_the_array():
    lib = binding.load_library(build_if_missing=True)
    A = torch.zeros(4096, 4096, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(4096, 4096, dtype=torch.bfloat16, device="cuda")
    # 256 tiles x 4 splits x 256 KiB of partials per tile >> 8 MiB
    assert run_noalloc(lib, A, A, C, 4) == WORKSPACE
    assert run_noalloc(lib, A, A, C, 1) == 1  # split_k must be 2..16
