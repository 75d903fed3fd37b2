"""The allocation-free split-K entry point against the oracle.

bwgemm_run_splitk_noalloc serves callers that cannot call cudaMalloc (a
memory manager that already reserved the device, a fixed device footprint,
loops that must not risk the synchronisation cudaMalloc / cudaFree can
cause): its split-K scratch lives in a fixed array inside the library.  Here
its C must match the oracle (bit for bit on integer inputs, within the
tolerance of the other parity tests on N(0,1) inputs) and the plan API's C
with the same split, on two calls in a row (the second call finds the first
call's leftovers in the shared array).  It must also handle the shapes where
the bookkeeping of the array differs -- a split cut to one slice (K of one
64-wide block), K = 0 -- and refuse scratch beyond the array and operands
that are not memory of the current device.

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import oracle
from dense_gemm_blackwell_03_gb300 import binding
from dense_gemm_blackwell_03_gb300.workloads import bits_of, make_matrix
from parity import compare

pytestmark = pytest.mark.gpu

INVALID_ARG = 1
WORKSPACE = 7
DT = {"bf16": (binding.BF16, torch.bfloat16), "fp16": (binding.FP16, torch.float16)}


def run_noalloc(lib, A, B, C, split, dtype="bf16"):
    M, K = A.shape
    N = B.shape[0]
    stream = ctypes.c_void_p(int(torch.cuda.current_stream().cuda_stream))
    return lib.bwgemm_run_splitk_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                         A.stride(0), B.stride(0), C.stride(0), DT[dtype][0],
                                         split, stream)


@pytest.mark.parametrize("M,N,K,dist,split,dtype", [
    (256, 512, 1600, "int2", 3, "bf16"),     # CTA-pair tiles, exact integers
    (100, 384, 4096, "normal", 4, "bf16"),   # single-CTA tiles, ragged M, N(0,1) inputs
    (300, 264, 1000, "normal", 2, "fp16"),   # ragged M, N and K, fp16
    (200, 520, 2000, "int2", 5, "fp16"),     # fp16 exact integers, five slices
    (256, 512, 64, "int2", 4, "bf16"),       # one K block: the split is cut to one slice
])
def test_noalloc_matches_oracle_and_plan(M, N, K, dist, split, dtype):
    assert torch.cuda.is_available()
    lib = binding.load_library(build_if_missing=True)
    A = make_matrix(M, K, dist, dtype=dtype, seed=1200 + split, device="cuda")
    B = make_matrix(N, K, dist, dtype=dtype, seed=1300 + split, device="cuda")
    want = oracle.gemm(bits_of(A), bits_of(B), dtype)
    exact = dist == "int2"
    with binding.Plan(0, split_k=split) as plan:
        via_plan = bits_of(plan.gemm(A, B))
        assert plan.status() == 0
    for _ in range(2):  # two calls in a row share (and reuse) the fixed scratch
        C = torch.full((M, N), 5.0, dtype=DT[dtype][1], device="cuda")
        assert run_noalloc(lib, A, B, C, split, dtype) == 0
        torch.cuda.synchronize()
        got = bits_of(C)
        compare(got, want, dtype, K, exact=exact)
        compare(got, via_plan, dtype, K, exact=exact)


def test_noalloc_empty_sum_zero_fills():
    lib = binding.load_library(build_if_missing=True)
    A = torch.empty(64, 0, dtype=torch.bfloat16, device="cuda")
    B = torch.empty(96, 0, dtype=torch.bfloat16, device="cuda")
    C = torch.full((64, 96), 5.0, dtype=torch.bfloat16, device="cuda")
    stream = ctypes.c_void_p(int(torch.cuda.current_stream().cuda_stream))
    rc = lib.bwgemm_run_splitk_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), 64, 96, 0, 8, 8,
                                       C.stride(0), binding.BF16, 2, stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert bool((C == 0).all())


def test_noalloc_refuses_scratch_beyond_the_array():
    lib = binding.load_library(build_if_missing=True)
    A = torch.zeros(4096, 4096, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(4096, 4096, dtype=torch.bfloat16, device="cuda")
    # 256 tiles x 4 splits x 256 KiB of partials per tile >> 8 MiB
    assert run_noalloc(lib, A, A, C, 4) == WORKSPACE
    assert run_noalloc(lib, A, A, C, 1) == INVALID_ARG  # split_k must be 2..16


def test_noalloc_refuses_host_operands():
    lib = binding.load_library(build_if_missing=True)
    A = torch.zeros(256, 512, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    hB = torch.zeros(256, 512, dtype=torch.bfloat16).pin_memory()
    hC = torch.zeros(256, 256, dtype=torch.bfloat16).pin_memory()
    assert run_noalloc(lib, A, hB, C, 2) == INVALID_ARG
    assert run_noalloc(lib, A, A, hC, 2) == INVALID_ARG
    torch.cuda.synchronize()
