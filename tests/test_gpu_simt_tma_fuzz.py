"""Seeded random cases for the TMA-fed FP32 SIMT kernel, compared in full
with the oracle.

The kernel runs for FP32 problems of at least a wave of 128 x 128 tiles
whose A and B have 16-byte aligned bases and pitches.  Each case draws M and
N so that the tiles exceed one wave, a K from 1 up, pitch padding that keeps
A and B describable by TMA, a C pitch that does or does not allow 16-byte
stores, alpha and beta (beta = 0 with a NaN-filled C), so that M, N and K
tails, partial K slices and both store forms appear.  The case list is fixed
by its seed.
"""
import math

import numpy as np
import pytest
import torch

from tests import parity

pytestmark = pytest.mark.gpu


def _cases(n=10, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M = int(rng.integers(2049, 3200))
        N = int(rng.integers(2433, 3200))   # at least 17 x 20 tiles: more than a wave of 304
        K = int(round(math.exp(rng.uniform(0.0, math.log(1500)))))
        pad_a = (4 - K % 4) % 4 + 4 * int(rng.integers(0, 3))   # lda a multiple of 4
        pad_b = (4 - N % 4) % 4 + 4 * int(rng.integers(0, 2))   # ldb a multiple of 4
        pad_c = int(rng.choice([0, 1, 3, 4]))
        alpha = float(rng.choice([1.0, -0.5, 2.0, 0.75]))
        beta = float(rng.choice([0.0, 1.0, -0.75]))
        out.append(((M, N, K), (pad_a, pad_b, pad_c), alpha, beta))
    return out


CASES = _cases()


@pytest.mark.parametrize("case", CASES, ids=["%dx%dx%d-p%d_%d_%d-a%g-b%g" % (c[0] + c[1] + (c[2], c[3])) for c in CASES])
def test_simt_tma_case_matches_oracle(case):
    import dense_gemm_09_gb300 as dg
    (M, N, K), pad, alpha, beta = case
    A, B, C = parity.host_operands("f32", M, N, K, seed=M + 3 * N + 7 * K)
    Cin = torch.full_like(C, float("nan")) if beta == 0.0 else C
    got, _, _ = parity.run("f32", A, B, Cin, alpha, beta, pad=pad)
    assert dg.last_kernel().startswith("sgemm_simt_tma_"), dg.last_kernel()
    assert dg.device_status(clear=False) == dg.OK
    assert torch.isfinite(got).all()
    assert parity.worst_ratio("f32", got, A, B, C, alpha, beta) <= 1.0
