"""Operands and results with more than 2^31 elements, on the GPU.

The C ABI takes 64-bit sizes and leading dimensions, and the kernels index
in 64 bits: an operand whose element count passes 2^31 must not wrap.  Each
case makes one operand (A, B or C) just over 2^31 elements and runs one
kernel family: the CTA-pair kernel on TMA (FP16 TN, TF32), the FP32 SIMT
kernel, and the producers for pitches TMA cannot describe (odd K: the TF32
cp.async producer and the 16-bit register-path producer).

Entries are seeded integers in {-1, 0, 1}, so every path is exact (sums of at
most K = 16384 such products stay far below 2^24, and below 2048 in
magnitude for the FP16 output with overwhelming probability).  Sampled
output rows (large A or C) or columns (large B) are compared with the oracle
bit for bit.  The oracle evaluates the sub-problem those rows or columns
define, on operands widened from the same host values that were copied to
the device.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests import parity

pytestmark = pytest.mark.gpu

BIG = 2**31

# (path, M, N, K, the operand past 2^31 elements, kernel name fragment)
CASES = [
    ("f16_tn", 131328, 512, 16384, "A", "_pair_"),
    ("f16_tn", 512, 131328, 16384, "B", "_pair_"),
    ("tf32", 131328, 512, 16384, "A", "_pair_"),
    ("tf32", 512, 16384, 131328, "B", "_pair_"),
    ("f32", 131328, 512, 16384, "A", "sgemm_simt"),
    ("f16_tn", 46400, 46400, 64, "C", "_pair_"),
    ("f32", 46400, 46400, 64, "C", "sgemm_simt"),
    ("tf32", 131100, 256, 16383, "A", "_cpasync"),
    ("f16_tn", 131100, 256, 16383, "A", "_ldst"),
]


def _ids(c):
    return "%s-%dx%dx%d-%s" % (c[0], c[1], c[2], c[3], c[4])


@pytest.mark.parametrize("path,M,N,K,big,kernel", CASES, ids=[_ids(c) for c in CASES])
def test_operand_past_2_31_elements(path, M, N, K, big, kernel):
    import dense_gemm_09_gb300 as dg
    tn = parity.is_tn(path)
    dt = parity.dtype(path)
    bshape = (N, K) if tn else (K, N)
    sizes = {"A": M * K, "B": bshape[0] * bshape[1], "C": M * N}
    assert sizes[big] > BIG
    g = si.generator(1000 + M % 997)
    A8 = si.small_integers_i8((M, K), g)
    B8 = si.small_integers_i8(bshape, g)
    C8 = si.small_integers_i8((M, N), g)
    dA = A8.cuda().to(dt)
    dB = B8.cuda().to(dt)
    dC = C8.cuda().to(dt)
    alpha, beta = 1.0, -1.0
    parity.fn(path)(dA, dB, dC, alpha, beta)
    torch.cuda.synchronize()
    assert dg.device_status() == dg.OK
    assert kernel in dg.last_kernel(), dg.last_kernel()
    del dA, dB

    kind = parity.oracle_kind(path)
    ck = kind if kind in ("f16", "bf16") else "f32"

    def wide(t8, k, trans=False):
        t = t8.to(dt)
        return oracle.widen(k, parity.np_operand(t), trans=trans)

    sel = np.unique(np.concatenate([si.boundary_indices(M if big != "B" else N),
                                    si.sample_positions(M if big != "B" else N, 1, 12, seed=77)[0]]))
    if big in ("A", "C"):
        # sampled rows (the high ones sit past element 2^31 of A or of C)
        # against all of B: the oracle's sub-problem on those rows of A and C
        rows = torch.as_tensor(sel)
        A64 = wide(A8[rows], kind)
        B64 = wide(B8, kind, trans=tn)
        C64 = wide(C8[rows], ck)
        ref, _ = oracle.gemm(A64, B64, C64, alpha, beta)
        got = dC[rows.cuda()].double().cpu().numpy()
    else:
        # sampled output columns: rows of the stored N x K B, or columns of K x N
        cols = torch.as_tensor(sel)
        A64 = wide(A8, kind)
        if tn:
            B64 = wide(B8[cols], kind, trans=True)
        else:
            B64 = wide(B8[:, cols].contiguous(), kind)
        C64 = wide(C8[:, cols].contiguous(), ck)
        ref, _ = oracle.gemm(A64, B64, C64, alpha, beta)
        got = dC[:, cols.cuda()].double().cpu().numpy()
    assert got.shape == ref.shape
    bad = np.flatnonzero(got.ravel() != ref.ravel())
    assert bad.size == 0, "%d mismatches, first at %d: got %r want %r" % (
        bad.size, bad[0], got.ravel()[bad[0]], ref.ravel()[bad[0]])
