"""Seeded synthetic inputs for the dense GEMM ``C = A @ B.T``.

This module only draws random numbers; it holds none of the GEMM's arithmetic
and is the one module shared by the CUDA path's tests and benchmark and by
the CPU oracle's checks.

Shapes follow the pages' workloads:
  * 4096^3 square reference point ("Writing a Blackwell GEMM by hand: 164 to
    1400 TFLOP/s", measurement section; the Blackwell deep dive's results
    list, all at 4096 x 4096 x 4096);
  * Llama-3-70B linears: prefill M=8192 (attention out N=K=8192, MLP up
    N=28672 K=8192) and decode M=256 (attention out, fused QKV N=10240,
    MLP up, MLP down N=8192 K=28672) (the CuTeDSL post, "two workloads, not
    one" section);
  * Gemma-3-27B-like 512 x 8192 x 5376 (the deep dive's production-shape
    experiment), and decode batches M in {1, 16, 64, 200} on an 8192 x 8192
    weight (the CuTeDSL post's note that real decode batches are 1 to 64).

Value distributions: activations i.i.d. N(0, 1); weights N(0, 0.02^2);
the square shape scales both operands by 1/sqrt(K); the bit-exact case draws
integers uniformly from {-2, ..., 2}.  Every tensor is drawn in fp32 by a
``torch.Generator`` seeded per shape and then rounded to bf16 / fp16.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

SEED_BASE = 20261202
INT_SEED_OFFSET = 1000

TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclass(frozen=True)
class Shape:
    name: str
    M: int
    N: int
    K: int
    a_dist: str  # "normal" | "normal_rsqrtk" | "int2"
    b_dist: str  # "normal" | "normal_rsqrtk" | "weight" | "int2"
    dtype: str = "bf16"
    group: int = 0  # index of the workload family (seed offset)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        """A and B read once, C written once (2-byte elements)."""
        return 2 * (self.M * self.K + self.N * self.K + self.M * self.N)

    def with_dtype(self, dtype: str) -> "Shape":
        return replace(self, dtype=dtype, name=f"{self.name}_{dtype}")


_ALL = [
    # family 0: 512^3 (N(0,1) and the bit-exact integer case)
    Shape("square512", 512, 512, 512, "normal", "normal", group=0),
    Shape("square512_int", 512, 512, 512, "int2", "int2", group=0),
    # family 1: 4096^3 square reference point, both operands N(0,1)/sqrt(K)
    Shape("square4096", 4096, 4096, 4096, "normal_rsqrtk", "normal_rsqrtk", group=1),
    Shape("square4096_fp16", 4096, 4096, 4096, "normal_rsqrtk", "normal_rsqrtk",
          dtype="fp16", group=1),
    # family 2: Llama-3-70B prefill linears, M = 8192 tokens
    Shape("prefill_attn_out", 8192, 8192, 8192, "normal", "weight", group=2),
    Shape("prefill_mlp_up", 8192, 28672, 8192, "normal", "weight", group=2),
    # family 3: Llama-3-70B decode linears, M = 256
    Shape("decode_attn_out", 256, 8192, 8192, "normal", "weight", group=3),
    Shape("decode_qkv", 256, 10240, 8192, "normal", "weight", group=3),
    Shape("decode_mlp_up", 256, 28672, 8192, "normal", "weight", group=3),
    Shape("decode_mlp_down", 256, 8192, 28672, "normal", "weight", group=3),
    # family 4: irregular / tail shapes
    Shape("gemma_512x8192x5376", 512, 8192, 5376, "normal", "weight", group=4),
    Shape("tail_m1", 1, 8192, 8192, "normal", "weight", group=4),
    Shape("tail_m16", 16, 8192, 8192, "normal", "weight", group=4),
    Shape("tail_m64", 64, 8192, 8192, "normal", "weight", group=4),
    Shape("tail_m200", 200, 8192, 8192, "normal", "weight", group=4),
]

SHAPES = {s.name: s for s in _ALL}


def seed_for(shape: Shape) -> int:
    seed = SEED_BASE + shape.group
    if shape.a_dist == "int2":
        seed += INT_SEED_OFFSET
    return seed


def _draw(rows: int, cols: int, dist: str, K: int, gen: torch.Generator, device,
          dtype: torch.dtype, ld: int | None) -> torch.Tensor:
    ld = cols if ld is None else ld
    if ld < cols:
        raise ValueError("leading dimension smaller than the row length")
    if dist == "int2":
        full = torch.randint(-2, 3, (rows, ld), generator=gen, device=device,
                             dtype=torch.int32).to(torch.float32)
    else:
        full = torch.randn((rows, ld), generator=gen, device=device, dtype=torch.float32)
        if dist == "normal_rsqrtk":
            full.mul_(1.0 / float(K) ** 0.5)
        elif dist == "weight":
            full.mul_(0.02)
        elif dist != "normal":
            raise ValueError(f"unknown distribution {dist!r}")
    out = full.to(dtype)
    del full
    return out[:, :cols] if ld != cols else out


def make_inputs(shape: Shape, device="cpu", seed: int | None = None,
                lda: int | None = None, ldb: int | None = None):
    """Return ``(A, B)``: A is M x K, B is N x K, both K-major (row stride lda/ldb)."""
    dtype = TORCH_DTYPES[shape.dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed_for(shape) if seed is None else seed)
    A = _draw(shape.M, shape.K, shape.a_dist, shape.K, gen, device, dtype, lda)
    B = _draw(shape.N, shape.K, shape.b_dist, shape.K, gen, device, dtype, ldb)
    return A, B


def make_matrix(rows: int, cols: int, dist: str, dtype: str = "bf16", device="cpu",
                seed: int = SEED_BASE, K: int | None = None, ld: int | None = None):
    """One seeded matrix (for ad-hoc edge-case shapes in the tests)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return _draw(rows, cols, dist, K if K is not None else cols, gen, device,
                 TORCH_DTYPES[dtype], ld)


def bits_of(t: torch.Tensor):
    """Raw 16-bit patterns of a bf16 / fp16 tensor as a host numpy uint16 array."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
