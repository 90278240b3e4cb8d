"""Seeded synthetic inputs for the GEMM workloads.

This module only draws numbers: it holds none of the GEMM arithmetic.  The
same host buffers it returns are handed both to the CUDA library (after a
copy to the device) and to the CPU oracle, so both sides see identical
operands.

Recipes (one torch CPU generator per problem, drawn in the order A, B, C):
  * uniform:  ``torch.rand(shape) * 2 - 1`` in float32 -> entries in [-1, 1);
  * normal-over-sqrt-K (the FP16 square sweep): ``torch.randn(shape) / sqrt(K)``
    then rounded to float16 (round-to-nearest-even, torch's conversion);
  * uniform rounded to float16 (the skinny FP16 case).
Sample positions for large problems come from a separate generator seeded
1234: 4096 (i, j) pairs uniform over [0, M) x [0, N), plus full rows and
columns at tile boundaries (0, 1, 63, 64, 127, 128, 129, 255, 256, M/2,
M-129, M-128, M-2, M-1), which covers 64/128/256-wide tiles and the last
partial tile whatever tile shape a kernel uses.

The workloads follow the pages' benchmark shapes: square FP32 problems with
alpha/beta ("如何优化一个 CUDA Matmul Kernel ... Worklog", 4092^2), the
8192 x 8192 x 4096 FP32 / TF32 table ("SGEMM CUDA代码学习", opening table),
the FP16 TN square sweep 2048..16384 ("HGEMM SMEM Swizzle 代码学习", opening
table) and ragged / skinny shapes that are not tile multiples.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    path: str          # "f32" (SIMT and TF32 share FP32 operands) or "f16_tn"
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    dist: str          # "uniform", "normal_sqrtk", "uniform_f16"
    c_zero: bool = False
    seed: int = 0


WORKLOADS = {
    w.name: w for w in [
        Workload("f32_256", "f32", 256, 256, 256, 1.0, 0.5, "uniform"),
        Workload("f32_4092", "f32", 4092, 4092, 4092, 0.5, 3.0, "uniform"),
        Workload("f32_8192x8192x4096", "f32", 8192, 8192, 4096, 1.0, 0.0, "uniform", c_zero=True),
        Workload("f32_8191x8193x4095", "f32", 8191, 8193, 4095, 1.5, -0.25, "uniform"),
        Workload("f16_tn_2048", "f16_tn", 2048, 2048, 2048, 1.0, 0.0, "normal_sqrtk", c_zero=True),
        Workload("f16_tn_4096", "f16_tn", 4096, 4096, 4096, 1.0, 0.0, "normal_sqrtk", c_zero=True),
        Workload("f16_tn_8192", "f16_tn", 8192, 8192, 8192, 1.0, 0.0, "normal_sqrtk", c_zero=True),
        Workload("f16_tn_12288", "f16_tn", 12288, 12288, 12288, 1.0, 0.0, "normal_sqrtk", c_zero=True),
        Workload("f16_tn_16384", "f16_tn", 16384, 16384, 16384, 1.0, 0.0, "normal_sqrtk", c_zero=True),
        Workload("f16_tn_8192x8192x4096", "f16_tn", 8192, 8192, 4096, 1.0, 0.0, "normal_sqrtk", c_zero=True),
        Workload("f16_tn_127x12288x4096", "f16_tn", 127, 12288, 4096, 1.5, -0.25, "uniform_f16"),
    ]
}


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def uniform(shape, g: torch.Generator) -> torch.Tensor:
    """float32 entries uniform in [-1, 1)."""
    return torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0


def small_integers(shape, g: torch.Generator, bound: int = 4, dtype=torch.float32) -> torch.Tensor:
    """Integers in [-bound, bound], exactly representable in every operand type."""
    return torch.randint(-bound, bound + 1, shape, generator=g).to(dtype)


def small_integers_i8(shape, g: torch.Generator, bound: int = 1) -> torch.Tensor:
    """Integers in [-bound, bound] as int8 (one byte each: operands of more
    than 2^31 elements stay a few GB on the host)."""
    return torch.randint(-bound, bound + 1, shape, generator=g, dtype=torch.int8)


def make(w: Workload, seed: int | None = None, pin: bool = False):
    """Host operands (A, B, C) for workload ``w``.

    f32 path: A (M, K), B (K, N), C (M, N), float32.
    f16_tn path: A (M, K), B (N, K) -- the TN store -- and C (M, N), float16.
    """
    g = generator(w.seed if seed is None else seed)
    M, N, K = w.M, w.N, w.K
    if w.path == "f32":
        A = uniform((M, K), g)
        B = uniform((K, N), g)
        C = torch.zeros((M, N), dtype=torch.float32) if w.c_zero else uniform((M, N), g)
    else:
        if w.dist == "normal_sqrtk":
            s = 1.0 / math.sqrt(K)
            A = (torch.randn((M, K), generator=g, dtype=torch.float32) * s).half()
            B = (torch.randn((N, K), generator=g, dtype=torch.float32) * s).half()
        else:
            A = uniform((M, K), g).half()
            B = uniform((N, K), g).half()
        C = torch.zeros((M, N), dtype=torch.float16) if w.c_zero else uniform((M, N), g).half()
    if pin:
        A, B, C = A.pin_memory(), B.pin_memory(), C.pin_memory()
    return A, B, C


def boundary_indices(n: int) -> np.ndarray:
    """Row (or column) indices at tile boundaries, deduplicated, in [0, n)."""
    cand = [0, 1, 63, 64, 127, 128, 129, 255, 256, n // 2, n - 129, n - 128, n - 2, n - 1]
    return np.array(sorted({c for c in cand if 0 <= c < n}), dtype=np.int64)


def sample_positions(M: int, N: int, count: int = 4096, seed: int = 1234):
    """``count`` seeded (i, j) positions uniform over [0, M) x [0, N)."""
    g = generator(seed)
    i = torch.randint(0, M, (count,), generator=g, dtype=torch.int64).numpy()
    j = torch.randint(0, N, (count,), generator=g, dtype=torch.int64).numpy()
    return i, j
