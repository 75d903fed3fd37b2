"""Pins for the CPU oracle (no GPU).

The oracle is the plain definition of the pages' GEMM (C = A * B^T, B stored
N x K; "Matrix Multiplication on NVIDIA's Blackwell", matmul definition and
the naive Kernel 1 listing) in fp64 with one final round-to-nearest-even.
Nothing here re-types its formula: every check compares it with something
fixed independently of it --

  * decoding: torch's own bf16/fp16 -> fp64 conversion of all 65536 patterns;
  * rounding: hand-derived fixtures under tests/golden/, numpy's float16
    conversion, torch's fp32 -> bf16 conversion (where the double is an fp32);
  * GEMM: identity and permutation matrices (result is a copy of A), rank-1
    products with closed-form sums, brute force in exact rational arithmetic
    with an independent table-based rounding, an fp64 numpy matmul;
  * host logic: row/column sub-blocks, strided operands, empty and K = 0 cases.

The last test plants mistakes in copies of oracle.c and checks that the pins
catch every one of them.
"""
from __future__ import annotations

import bisect
import os
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_blackwell_03_gb300.workloads import bits_of, make_matrix

TORCH16 = {"bf16": torch.bfloat16, "fp16": torch.float16}
FMT = {"bf16": (7, 8, 127), "fp16": (10, 5, 15)}  # significand bits, exponent bits, bias


# --------------------------------------------------------------------------
# independent helpers (torch decoding, exact rationals)
# --------------------------------------------------------------------------
def torch_decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(TORCH16[dtype]).to(torch.float64).numpy()


class TableRounding:
    """Round exact rationals by searching the sorted list of every finite
    positive value of the format (decoded by torch), ties to the even pattern;
    +inf is treated as the successor of the largest finite value."""

    def __init__(self, dtype: str):
        mant, _, bias = FMT[dtype]
        bits = np.arange(0, 0x8000, dtype=np.uint16)
        vals = torch_decode(bits, dtype)
        keep = np.isfinite(vals)
        pairs = sorted(zip(vals[keep].tolist(), bits[keep].tolist()))
        self.values = [Fraction(v) for v, _ in pairs]
        self.bits = [b for _, b in pairs]
        inf_bits = ((1 << FMT[dtype][1]) - 1) << mant
        self.values.append(Fraction(2) ** (bias + 1))  # max + one ulp
        self.bits.append(inf_bits)

    def __call__(self, x: Fraction) -> int:
        sign = 0x8000 if x < 0 else 0
        a = -x if x < 0 else x
        if a >= self.values[-1]:
            return sign | self.bits[-1]
        i = bisect.bisect_right(self.values, a) - 1
        lo, hi = self.values[i], self.values[i + 1]
        if a == lo:
            return sign | self.bits[i]
        mid = (lo + hi) / 2
        if a < mid:
            pick = i
        elif a > mid:
            pick = i + 1
        else:
            pick = i if self.bits[i] % 2 == 0 else i + 1
        return sign | self.bits[pick]


def load_fixtures(path):
    xs, want = [], []
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            v, b = line.split()[:2]
            xs.append(float.fromhex(v))
            want.append(int(b, 16))
    return np.array(xs, dtype=np.float64), np.array(want, dtype=np.uint16)


def random_bits(rng: np.random.Generator, shape, dtype: str, exp_lo: int, exp_hi: int):
    """Random finite patterns with unbiased exponents in [exp_lo, exp_hi]
    (exp_lo below the normal range gives subnormals)."""
    mant, ebits, bias = FMT[dtype]
    n = int(np.prod(shape))
    sign = rng.integers(0, 2, n)
    e = rng.integers(exp_lo, exp_hi + 1, n)
    m = rng.integers(0, 1 << mant, n)
    field = np.clip(e + bias, 0, (1 << ebits) - 2)
    out = (sign << 15) | (field << mant) | m
    return out.astype(np.uint16).reshape(shape)


# --------------------------------------------------------------------------
# the pin battery (each takes an Oracle instance; also run against mutants)
# --------------------------------------------------------------------------
def pin_decode(orc, dtype):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.decode(bits, dtype)
    want = torch_decode(bits, dtype)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def pin_round_fixtures(orc, dtype, golden_dir):
    xs, want = load_fixtures(os.path.join(golden_dir, f"round_{dtype}.txt"))
    got = orc.round_to(xs, dtype)
    bad = [(x.hex(), hex(g), hex(w)) for x, g, w in zip(xs, got, want) if g != w]
    assert not bad, f"rounding fixtures disagree: {bad}"


def pin_round_library(orc, dtype):
    rng = np.random.default_rng(7)
    # doubles spread over the whole range of the format, plus exact ties
    mant, _, bias = FMT[dtype]
    e = rng.integers(-bias - mant - 2, bias + 2, 20000)
    x = np.ldexp(rng.uniform(1.0, 2.0, e.size), e) * rng.choice([-1.0, 1.0], e.size)
    ties = np.ldexp((2.0 * rng.integers(1 << mant, 1 << (mant + 1), 4000) + 1.0),
                    rng.integers(-bias - mant, bias - mant, 4000) - 1)
    x = np.concatenate([x, ties, -ties])
    got = orc.round_to(x, dtype)
    if dtype == "fp16":
        with np.errstate(over="ignore"):  # overflow to inf is part of the check
            want = x.astype(np.float16).view(np.uint16)  # numpy rounds double -> half directly
        assert np.array_equal(got, want)
    # torch rounds fp32 -> bf16 / fp16 with ties-to-even: compare where x is an fp32
    x32 = x.astype(np.float32)
    exact = x32.astype(np.float64) == x
    t = torch.from_numpy(x32[exact]).to(TORCH16[dtype])
    want32 = bits_of(t)
    assert np.array_equal(got[exact], want32)


def pin_identity(orc, dtype):
    A = bits_of(make_matrix(37, 96, "normal", dtype, seed=11))
    eye = bits_of(torch.eye(96, dtype=TORCH16[dtype]))
    C = orc.gemm(A, eye, dtype)
    assert np.array_equal(C, A)


def pin_permutation(orc, dtype):
    A = bits_of(make_matrix(19, 80, "normal", dtype, seed=12))
    perm = np.random.default_rng(3).permutation(80)
    P = torch.zeros(80, 80, dtype=TORCH16[dtype])
    P[torch.arange(80), torch.from_numpy(perm)] = 1  # row j of B is e_perm[j]
    C = orc.gemm(A, bits_of(P), dtype)
    assert np.array_equal(C, A[:, perm])


def pin_rank1(orc, dtype):
    # A[i,k] = u_i a_k, B[j,k] = v_j b_k  =>  C[i,j] = u_i v_j S, S = sum_k a_k b_k.
    # a_k = k mod 3 and b_k = (k mod 5) - 1: (k mod 3, k mod 5) runs through all
    # 15 pairs once per period, so a period contributes (0+1+2) * (-1+0+1+2+3) = 15
    # and S = 15 * (K // 15) + (sum of the first K mod 15 terms).
    K = 15 * 8 + 7
    a = np.array([k % 3 for k in range(K)], dtype=np.float64)
    b = np.array([(k % 5) - 1 for k in range(K)], dtype=np.float64)
    S = 15 * (K // 15) + sum((k % 3) * ((k % 5) - 1) for k in range(K % 15))
    assert S == 123
    u = np.array([1.0, -2.0, 0.5, 4.0, -0.25, 8.0])
    v = np.array([-1.0, 2.0, 0.125, -16.0, 1.0])
    A = torch.from_numpy(np.outer(u, a)).to(TORCH16[dtype])
    B = torch.from_numpy(np.outer(v, b)).to(TORCH16[dtype])
    C = orc.gemm(bits_of(A), bits_of(B), dtype)
    # u_i v_j S = (power of two) * 123 is exactly representable in both formats
    want = bits_of(torch.from_numpy(np.outer(u, v) * S).to(TORCH16[dtype]))
    assert np.array_equal(C, want)


def pin_rank1_rounded(orc, dtype):
    # all-ones rows: S = K; K = 2^(mant+1) + 1 sits exactly halfway between two
    # representable integers and must round to the even one, 2^(mant+1).
    mant = FMT[dtype][0]
    K = (1 << (mant + 1)) + 1
    A = torch.ones(3, K, dtype=TORCH16[dtype])
    B = torch.ones(2, K, dtype=TORCH16[dtype])
    C = orc.gemm(bits_of(A), bits_of(B), dtype)
    want = bits_of(torch.full((3, 2), float(K - 1), dtype=TORCH16[dtype]))
    assert np.array_equal(C, want)
    # K = 2^(mant+1) + 3: halfway between K - 1 and K + 1, the even one is K + 1
    K = (1 << (mant + 1)) + 3
    C = orc.gemm(bits_of(torch.ones(1, K, dtype=TORCH16[dtype])),
                 bits_of(torch.ones(1, K, dtype=TORCH16[dtype])), dtype)
    assert C[0, 0] == bits_of(torch.tensor([float(K + 1)], dtype=TORCH16[dtype]))[0]


def pin_bruteforce(orc, dtype, trials=60):
    rnd = TableRounding(dtype)
    rng = np.random.default_rng(99)
    mant, _, bias = FMT[dtype]
    for t in range(trials):
        M, N, K = (int(x) for x in rng.integers(1, 9, 3))
        if t % 3 == 0:
            lo, hi = -bias - mant, -bias + 3  # subnormal and tiny results
        elif t % 3 == 1:
            lo, hi = -3, 3
        else:
            lo, hi = bias // 2 - 2, bias // 2 + 1  # sums near or past overflow
        A = random_bits(rng, (M, K), dtype, lo, hi)
        B = random_bits(rng, (N, K), dtype, lo, hi)
        av = [[Fraction(float(x)) for x in row] for row in torch_decode(A, dtype)]
        bv = [[Fraction(float(x)) for x in row] for row in torch_decode(B, dtype)]
        C = orc.gemm(A, B, dtype)
        for i in range(M):
            for j in range(N):
                s = sum((av[i][k] * bv[j][k] for k in range(K)), Fraction(0))
                want = rnd(s)
                assert C[i, j] == want, (dtype, t, i, j, hex(C[i, j]), hex(want))


def pin_numpy_fp64(orc, dtype):
    A = bits_of(make_matrix(33, 300, "normal", dtype, seed=21))
    B = bits_of(make_matrix(41, 300, "weight", dtype, seed=22))
    _, acc = orc.gemm(A, B, dtype, with_acc=True)
    ref = torch_decode(A, dtype) @ torch_decode(B, dtype).T
    assert np.linalg.norm(acc - ref) <= 1e-12 * np.linalg.norm(ref)


def pin_subblock(orc, dtype):
    A = bits_of(make_matrix(50, 64, "normal", dtype, seed=31))
    B = bits_of(make_matrix(70, 64, "normal", dtype, seed=32))
    full = orc.gemm(A, B, dtype)
    rows = [49, 0, 7, 7, 23]
    cols = [3, 69, 0, 41]
    assert np.array_equal(orc.gemm(A, B, dtype, rows=rows), full[rows])
    assert np.array_equal(orc.gemm(A, B, dtype, cols=cols), full[:, cols])
    assert np.array_equal(orc.gemm(A, B, dtype, rows=rows, cols=cols), full[np.ix_(rows, cols)])


PINS = [
    ("decode", lambda o, d, g: pin_decode(o, d)),
    ("round_fixtures", lambda o, d, g: pin_round_fixtures(o, d, g)),
    ("round_library", lambda o, d, g: pin_round_library(o, d)),
    ("identity", lambda o, d, g: pin_identity(o, d)),
    ("permutation", lambda o, d, g: pin_permutation(o, d)),
    ("rank1", lambda o, d, g: pin_rank1(o, d)),
    ("rank1_rounded", lambda o, d, g: pin_rank1_rounded(o, d)),
    ("bruteforce", lambda o, d, g: pin_bruteforce(o, d, trials=24)),
    ("numpy_fp64", lambda o, d, g: pin_numpy_fp64(o, d)),
    ("subblock", lambda o, d, g: pin_subblock(o, d)),
]


# --------------------------------------------------------------------------
# tests on the real oracle
# --------------------------------------------------------------------------
@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_decode_matches_torch(orc, dtype):
    pin_decode(orc, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_round_golden_fixtures(orc, dtype, golden_dir):
    pin_round_fixtures(orc, dtype, golden_dir)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_round_matches_library_conversions(orc, dtype):
    pin_round_library(orc, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_identity(orc, dtype):
    pin_identity(orc, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_permutation(orc, dtype):
    pin_permutation(orc, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_rank1_closed_form(orc, dtype):
    pin_rank1(orc, dtype)
    pin_rank1_rounded(orc, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_bruteforce_exact_rationals(orc, dtype):
    pin_bruteforce(orc, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fp64_sums_match_numpy(orc, dtype):
    pin_numpy_fp64(orc, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_row_col_subblocks(orc, dtype):
    pin_subblock(orc, dtype)


def test_integer_inputs_are_exact(orc):
    # integer entries in {-2..2}: every partial sum is an integer of magnitude
    # <= 4K, so the fp64 sum is exact; compare with integer arithmetic.
    A = make_matrix(64, 512, "int2", "bf16", seed=41)
    B = make_matrix(48, 512, "int2", "bf16", seed=42)
    _, acc = orc.gemm(bits_of(A), bits_of(B), "bf16", with_acc=True)
    exact = A.to(torch.int64) @ B.to(torch.int64).T
    assert np.array_equal(acc, exact.numpy().astype(np.float64))


def test_strided_operands(orc):
    A = make_matrix(20, 72, "normal", "bf16", seed=51, ld=96)  # lda = 96 > K = 72
    B = make_matrix(30, 72, "normal", "bf16", seed=52, ld=80)
    a_full = bits_of(A.as_strided((20, 96), (96, 1)))  # padded rows as stored
    b_full = bits_of(B.as_strided((30, 80), (80, 1)))
    got = orc.gemm(a_full[:, :72], b_full[:, :72], "bf16")
    want = orc.gemm(np.ascontiguousarray(a_full[:, :72]), np.ascontiguousarray(b_full[:, :72]), "bf16")
    assert np.array_equal(got, want)


def test_degenerate_shapes(orc):
    A = bits_of(make_matrix(5, 0, "normal", "bf16"))
    B = bits_of(make_matrix(7, 0, "normal", "bf16"))
    C = orc.gemm(A, B, "bf16")  # K = 0: the empty sum is +0
    assert C.shape == (5, 7) and not C.any()
    assert orc.gemm(np.zeros((0, 8), np.uint16), np.zeros((3, 8), np.uint16), "bf16").shape == (0, 3)
    assert orc.gemm(np.zeros((4, 8), np.uint16), np.zeros((0, 8), np.uint16), "bf16").shape == (4, 0)
    # an exact-zero sum of signed products is +0
    A = bits_of(torch.tensor([[2.0, -2.0, 0.0]], dtype=torch.bfloat16))
    B = bits_of(torch.tensor([[1.0, 1.0, -3.0]], dtype=torch.bfloat16))
    assert orc.gemm(A, B, "bf16")[0, 0] == 0x0000


def test_rejects_bad_arguments(orc):
    A = np.zeros((4, 8), np.uint16)
    with pytest.raises(ValueError):
        orc.gemm(A, np.zeros((3, 9), np.uint16), "bf16")
    with pytest.raises(ValueError):
        orc.gemm(A, A, "fp8")
    with pytest.raises(ValueError):
        orc.gemm(A, A, "bf16", rows=[4])


def test_threads_do_not_change_results(orc):
    A = bits_of(make_matrix(64, 256, "normal", "bf16", seed=61))
    B = bits_of(make_matrix(40, 256, "normal", "bf16", seed=62))
    assert np.array_equal(orc.gemm(A, B, "bf16", threads=1), orc.gemm(A, B, "bf16", threads=0))


# --------------------------------------------------------------------------
# planted mistakes: each broken copy of oracle.c must fail at least one pin
# --------------------------------------------------------------------------
MUTANTS = {
    "ties_to_odd": ("fmod(fl, 2.0) != 0.0", "fmod(fl, 2.0) == 0.0"),
    "truncate": ("if (rem > 0.5 || (rem == 0.5", "if (0 && (rem == 0.5"),
    "drop_last_term": ("for (int64_t k = 0; k < K; ++k)\n                    s +=",
                       "for (int64_t k = 0; k + 1 < K; ++k)\n                    s +="),
    "wrong_sign": ("s += arow[k] * widen[brow[k]];", "s -= arow[k] * widen[brow[k]];"),
    "shifted_index": ("s += arow[k] * widen[brow[k]];",
                      "s += arow[k] * widen[brow[k > 0 ? k - 1 : 0]];"),
    "ignore_col_subset": ("const int64_t j = cols ? cols[c] : c;", "const int64_t j = c % N;"),
    "subnormal_exponent": ("ldexp((double)m, 1 - f.bias - f.mant_bits)",
                           "ldexp((double)m, -f.bias - f.mant_bits)"),
    "overflow_saturates": ("if (E > emax)\n            return (uint16_t)(sign | inf_bits);\n    }",
                           "if (E > emax)\n            return (uint16_t)(sign | (inf_bits - 1));\n    }"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, tmp_path, golden_dir):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant_c = tmp_path / f"oracle_{name}.c"
    mutant_c.write_text(src.replace(old, new))
    lib = tmp_path / f"liboracle_{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", str(mutant_c), "-o", str(lib),
                    "-lm"], check=True, capture_output=True)
    orc = oracle.Oracle(str(lib))
    caught = []
    for pin_name, pin in PINS:
        for dtype in ("bf16", "fp16"):
            try:
                pin(orc, dtype, golden_dir)
            except AssertionError:
                caught.append(f"{pin_name}/{dtype}")
    assert caught, f"no pin caught the planted mistake {name}"
