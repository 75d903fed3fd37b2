"""Comparison of the CUDA path's output with the oracle's (shared by the GPU tests,
``__graft_entry__.smoke`` and ``bench.py``'s parity spot check).

Tolerance for N(0,1)-type inputs (fp32 accumulation on the GPU against the
oracle's fp64 sum with one rounding):
  * normwise   ||C - C_ref||_F / ||C_ref||_F <= 4e-3, and
  * elementwise |C - C_ref| <= 2 ulp(C_ref) + 1e-3 * sqrt(K) * rms(C_ref),
where ulp is the spacing of the output format at the oracle's value (the
subnormal spacing below the smallest normal) and rms is over the compared
elements.  Integer inputs in {-2..2} must match bit for bit (exact zeros of
either sign count as equal: the sign of an exact-zero sum depends on the
order in which signed zero products are added).
"""
from __future__ import annotations

import numpy as np
import torch

FMT = {"bf16": (7, 127), "fp16": (10, 15)}  # significand bits, bias
TORCH16 = {"bf16": torch.bfloat16, "fp16": torch.float16}


def values(bits: np.ndarray, dtype: str) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(TORCH16[dtype]).to(torch.float64).numpy()


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    mant, bias = FMT[dtype]
    emin = 1 - bias
    a = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - mant).astype(np.int64))


def compare(got_bits: np.ndarray, ref_bits: np.ndarray, dtype: str, K: int, exact: bool = False):
    """Raise AssertionError with a summary when the tolerance is not met; return stats."""
    assert got_bits.shape == ref_bits.shape, (got_bits.shape, ref_bits.shape)
    g = values(got_bits, dtype)
    r = values(ref_bits, dtype)
    finite = np.isfinite(r)
    assert np.array_equal(np.isfinite(g), finite), "non-finite pattern differs"
    assert np.array_equal(g[~finite], r[~finite]) or not (~finite).any(), "inf sign differs"
    if exact:
        same = (got_bits == ref_bits) | ((g == 0) & (r == 0))
        bad = int((~same).sum())
        assert bad == 0, f"{bad} of {same.size} elements differ from the oracle bit pattern"
        return {"max_abs": 0.0, "rel_fro": 0.0, "bad": 0}
    g, r = g[finite], r[finite]
    diff = np.abs(g - r)
    nref = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(g - r) / nref) if nref > 0 else float(np.linalg.norm(g - r))
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    bound = 2.0 * ulp(r, dtype) + 1e-3 * np.sqrt(max(K, 1)) * rms
    bad = int((diff > bound).sum())
    stats = {"max_abs": float(diff.max()) if diff.size else 0.0, "rel_fro": rel, "bad": bad,
             "rms": rms}
    assert rel <= 4e-3, f"normwise relative error {rel:.3e} > 4e-3 ({stats})"
    assert bad == 0, f"{bad} elements outside 2 ulp + 1e-3*sqrt(K)*rms ({stats})"
    return stats


def sample_indices(n: int, count: int, seed: int, tile: int = 128) -> np.ndarray:
    """Seeded sample of `count` indices in [0, n): both ends and tile edges first."""
    must = {0, n - 1}
    for t in range(tile, n, tile * 7):
        must.update({t - 1, t})
    must = sorted(i for i in must if 0 <= i < n)[: count // 2]
    rng = np.random.default_rng(seed)
    rest = [i for i in rng.permutation(n)[: count * 2].tolist() if i not in must]
    idx = (must + rest)[:count]
    return np.array(sorted(set(idx)), dtype=np.int64)
