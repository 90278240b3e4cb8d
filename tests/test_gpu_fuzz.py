"""Seeded random cases across every path, compared in full with the oracle.

Each case draws a path, a shape (log-uniform sizes, so tiny, ragged and
multi-tile problems all appear), row-pitch padding and base offsets (which
decide between the TMA, cp.async, register-path and scalar kernels), alpha
and beta (beta = 0 with a NaN-filled C), and a tile configuration forced
through the tuning hook (the automatic choice, the CTA pair with whole tiles
or with the stream-K tail forced on, the wide pair, a single-CTA width,
split-K).  The case list is fixed by
its seed, so a failure reproduces.
"""
import math

import numpy as np
import pytest
import torch

from tests import parity

pytestmark = pytest.mark.gpu


def _cases(n=240, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        path = parity.PATHS[i % len(parity.PATHS)]
        M, N, K = (int(round(math.exp(rng.uniform(0.0, math.log(1400))))) for _ in range(3))
        pad = tuple(int(x) for x in rng.choice([0, 0, 0, 1, 3, 8], size=3))
        offset = tuple(int(x) for x in rng.choice([0, 0, 0, 0, 1, 2], size=3))
        alpha = float(rng.choice([1.0, -0.5, 2.0, 0.75]))
        beta = float(rng.choice([0.0, 1.0, -0.75]))
        if path == "f32":
            tune = (0, 256, 1)
        else:
            kind = int(rng.integers(0, 6))
            bn = int(rng.choice([64, 128, 192, 256]))
            split = int(rng.integers(2, 5))
            tune = {0: (0, 256, 1), 1: (1, 256, 1), 2: (2, bn, 1), 3: (3, bn, split),
                    4: (1, 256, 2), 5: (5, 256, 1)}[kind]
        out.append((path, (M, N, K), pad, offset, alpha, beta, tune))
    return out


CASES = _cases()


def _id(c):
    path, (M, N, K), pad, off, alpha, beta, tune = c
    return "%s-%dx%dx%d-p%d%d%d-o%d%d%d-a%g-b%g-t%d_%d_%d" % ((path, M, N, K) + pad + off + (alpha, beta) + tune)


@pytest.mark.parametrize("case", CASES, ids=[_id(c) for c in CASES])
def test_fuzz_case_matches_oracle(case):
    import dense_gemm_09_gb300 as dg
    path, (M, N, K), pad, offset, alpha, beta, tune = case
    A, B, C = parity.host_operands(path, M, N, K, seed=M * 7 + N * 13 + K)
    if tune[0] != 0:
        dg.tune_next(*tune)
    Cin = torch.full_like(C, float("nan")) if beta == 0.0 else C
    got, _, _ = parity.run(path, A, B, Cin, alpha, beta, pad=pad, offset=offset)
    assert dg.device_status(clear=False) == dg.OK
    assert torch.isfinite(got).all(), dg.last_kernel()
    assert parity.worst_ratio(path, got, A, B, C, alpha, beta) <= 1.0, dg.last_kernel()


# The small-M pair (tuning variant 8) on seeded random problems: one or two
# bands of rows, any N (most within one wave of pairs), pitch padding, base
# offsets and both betas.  Where the operands rule the kernel out (pitches
# TMA cannot describe, too many tiles) the call chooses another one; every
# result is compared in full with the oracle.
def _pair128_cases(n=48, seed=20261203):
    rng = np.random.default_rng(seed)
    paths = [p for p in parity.PATHS if p != "f32"]
    out = []
    for i in range(n):
        path = paths[i % len(paths)]
        M = int(rng.integers(1, 257))
        # N and K multiples of 8 and pads / offsets of 8 or 16 elements keep
        # the pitches and bases TMA-describable, so that this kernel runs;
        # one case in eight pads by 3 (another kernel must take it)
        N = 8 * math.ceil(math.exp(rng.uniform(math.log(64), math.log(6000))) / 8)
        K = 8 * math.ceil(math.exp(rng.uniform(math.log(16), math.log(1500))) / 8)
        pad = tuple(int(x) for x in rng.choice([0, 0, 0, 8, 16], size=3))
        if i % 8 == 7:
            pad = (3, 0, 0)
        offset = tuple(int(x) for x in rng.choice([0, 0, 0, 8], size=3))
        alpha = float(rng.choice([1.0, -0.5, 0.75]))
        beta = float(rng.choice([0.0, 1.0, -0.75]))
        bn = int(rng.choice([128, 192, 256]))
        out.append((path, (M, N, K), pad, offset, alpha, beta, (8, bn, 1)))
    return out


PAIR128_CASES = _pair128_cases()


@pytest.mark.parametrize("case", PAIR128_CASES, ids=[_id(c) for c in PAIR128_CASES])
def test_fuzz_pair128_matches_oracle(case):
    test_fuzz_case_matches_oracle(case)
