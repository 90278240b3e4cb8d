"""gemm_tf32_ws: operands TMA cannot load are copied into a caller workspace
with a padded pitch, then the TMA kernels run on the copies.

Checked on the GPU against the oracle (full comparison), and bit for bit
against gemm_tf32 on an aligned copy of the same operands -- the copy changes
no value, so the product must not change either.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from tests import parity

pytestmark = pytest.mark.gpu


def _operands(M, N, K, pad, offset, seed):
    A, B, C = parity.host_operands("tf32", M, N, K, seed=seed)
    dA, _ = parity.to_device_padded(A, pad[0], offset_elems=offset[0])
    dB, _ = parity.to_device_padded(B, pad[1], offset_elems=offset[1])
    return A, B, C, dA, dB


def _workspace(dg, dA, dB):
    n = dg.tf32_workspace_bytes(dA, dB)
    return n, (torch.empty(max(n, 1), dtype=torch.uint8, device="cuda") if n else None)


# (M, N, K, pitch padding (A, B), base offset in elements (A, B))
CASES = [
    (129, 257, 301, (0, 0), (0, 0)),       # odd K and N: both pitches off 16 bytes
    (300, 520, 1000, (1, 0), (0, 0)),      # A pitch 1001
    (300, 520, 1000, (0, 3), (0, 0)),      # B pitch 523
    (300, 520, 1000, (0, 0), (1, 2)),      # aligned pitches, bases off 16 bytes
    (1, 300, 703, (0, 0), (0, 0)),
    (700, 5, 300, (0, 1), (0, 0)),
    (1000, 1100, 513, (2, 2), (3, 1)),     # more tiles than SMs, both repacked
]


@pytest.mark.parametrize("M,N,K,pad,offset", CASES)
def test_ws_matches_oracle(M, N, K, pad, offset):
    import dense_gemm_09_gb300 as dg
    A, B, C, dA, dB = _operands(M, N, K, pad, offset, seed=M + N + K)
    n, ws = _workspace(dg, dA, dB)
    assert n > 0
    dC = C.cuda()
    dg.gemm_tf32_ws(dA, dB, dC, 1.5, -0.25, workspace=ws)
    torch.cuda.synchronize()
    assert dg.last_kernel().endswith("_tma"), dg.last_kernel()
    assert parity.worst_ratio("tf32", dC.cpu(), A, B, C, 1.5, -0.25) <= 1.0


@pytest.mark.parametrize("M,N,K,pad,offset", CASES)
def test_ws_bit_identical_to_aligned_copy(M, N, K, pad, offset):
    import dense_gemm_09_gb300 as dg
    A, B, C, dA, dB = _operands(M, N, K, pad, offset, seed=7 * M + K)
    _, ws = _workspace(dg, dA, dB)
    got = C.cuda()
    dg.gemm_tf32_ws(dA, dB, got, 0.75, 0.5, workspace=ws)
    # the same values in buffers TMA can load directly (pitches padded)
    Aa = torch.zeros((M, (K + 3) // 4 * 4), device="cuda")[:, :K]
    Ba = torch.zeros((K, (N + 3) // 4 * 4), device="cuda")[:, :N]
    Aa.copy_(dA)
    Ba.copy_(dB)
    want = C.cuda()
    dg.gemm_tf32(Aa, Ba, want, 0.75, 0.5)
    torch.cuda.synchronize()
    assert dg.last_kernel().endswith("_tma")
    assert torch.equal(got, want)


def test_ws_integers_bit_exact():
    import dense_gemm_09_gb300 as dg
    M, N, K = 257, 1031, 771
    A, B, C = parity.host_operands("tf32", M, N, K, seed=12, dist="int")
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    _, ws = _workspace(dg, dA, dB)
    dg.gemm_tf32_ws(dA, dB, dC, 1.0, 2.0, workspace=ws)
    ref, _ = parity.reference("tf32", A, B, C, 1.0, 2.0)
    assert np.array_equal(dC.cpu().double().numpy(), ref)


def test_ws_rejects_small_or_misaligned_workspace():
    import dense_gemm_09_gb300 as dg
    M, N, K = 64, 72, 301
    A, B, C, dA, dB = _operands(M, N, K, (0, 0), (0, 0), seed=3)
    n, ws = _workspace(dg, dA, dB)
    dC = C.cuda()
    with pytest.raises(dg.DgemmError) as e:
        dg.gemm_tf32_ws(dA, dB, dC, 1.0, 0.0, workspace=ws[: n - 16])
    assert e.value.status == dg.ERR_INVALID_ARG
    with pytest.raises(dg.DgemmError):
        dg.gemm_tf32_ws(dA, dB, dC, 1.0, 0.0, workspace=None)
    big = torch.empty(n + 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(dg.DgemmError):
        dg.gemm_tf32_ws(dA, dB, dC, 1.0, 0.0, workspace=big[4:])  # base off 16 bytes
    torch.cuda.synchronize()
    assert torch.equal(dC.cpu(), C)  # nothing was launched


def test_ws_not_needed_for_aligned_operands():
    import dense_gemm_09_gb300 as dg
    M, N, K = 300, 520, 1000
    A, B, C = parity.host_operands("tf32", M, N, K, seed=4)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    assert dg.tf32_workspace_bytes(dA, dB) == 0
    dg.gemm_tf32_ws(dA, dB, dC, 1.0, 0.5, workspace=None)
    torch.cuda.synchronize()
    assert parity.worst_ratio("tf32", dC.cpu(), A, B, C, 1.0, 0.5) <= 1.0


def test_ws_ragged_workload_full_size():
    # the FP32 8191 x 8193 x 4095 workload (alpha 1.5, beta -0.25) through
    # the TF32 tensor cores, both operands repacked
    import dense_gemm_09_gb300 as dg
    w = si.WORKLOADS["f32_8191x8193x4095"]
    A, B, C = si.make(w)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    n, ws = _workspace(dg, dA, dB)
    assert n > 0
    dg.gemm_tf32_ws(dA, dB, dC, w.alpha, w.beta, workspace=ws)
    torch.cuda.synchronize()
    assert dg.device_status() == dg.OK
    assert "_pair_" in dg.last_kernel()
    assert parity.sampled_check("tf32", dC, A, B, C, w.alpha, w.beta) <= 1.0


# gemm_f32_ws: the SIMT path with the same workspace.  B is copied when its
# rows rule out 16-byte loads; A is copied too when the problem has at least
# a wave of tiles (then the TMA-fed kernel runs), and otherwise stays in place.
F32_CASES = [
    (129, 257, 301, (0, 0), (0, 0)),      # odd N: B's pitch off 16 bytes
    (300, 520, 1000, (0, 3), (0, 0)),     # B pitch 523
    (300, 520, 1000, (0, 0), (0, 2)),     # B base off 16 bytes
    (1000, 1100, 513, (2, 2), (3, 1)),
    (2100, 2500, 301, (0, 0), (0, 0)),    # a wave of tiles: A (pitch 301) and B (2500 ok) -> A copied
    (2049, 2561, 300, (1, 0), (0, 0)),    # a wave of tiles: A pitch 301, B pitch 2561: both copied
]


@pytest.mark.parametrize("M,N,K,pad,offset", F32_CASES)
def test_f32_ws_matches_oracle_and_plain_call(M, N, K, pad, offset):
    import dense_gemm_09_gb300 as dg
    A, B, C = parity.host_operands("f32", M, N, K, seed=5 * M + N)
    dA, _ = parity.to_device_padded(A, pad[0], offset_elems=offset[0])
    dB, _ = parity.to_device_padded(B, pad[1], offset_elems=offset[1])
    n, ws = _workspace(dg, dA, dB)
    assert n > 0
    got = C.cuda()
    dg.gemm_f32_ws(dA, dB, got, 1.5, -0.25, workspace=ws)
    torch.cuda.synchronize()
    # B now loads in 16-byte pieces, or both operands by TMA when the problem
    # has at least a wave of tiles
    big = ((M + 127) // 128) * ((N + 127) // 128) >= 304
    if big:
        assert dg.last_kernel().startswith("sgemm_simt_tma_"), dg.last_kernel()
    else:
        assert not dg.last_kernel().endswith("cpasync4"), dg.last_kernel()
    assert parity.worst_ratio("f32", got.cpu(), A, B, C, 1.5, -0.25) <= 1.0
    # the same FP32 FMAs in the same order as the plain call on the same values
    want = C.cuda()
    dg.gemm_f32(dA, dB, want, 1.5, -0.25)
    torch.cuda.synchronize()
    assert torch.equal(got, want)


def test_f32_ws_rejects_a_missing_workspace():
    import dense_gemm_09_gb300 as dg
    A, B, C = parity.host_operands("f32", 64, 77, 40, seed=1)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    assert dg.tf32_workspace_bytes(dA, dB) > 0
    with pytest.raises(dg.DgemmError) as e:
        dg.gemm_f32_ws(dA, dB, dC, 1.0, 0.0, workspace=None)
    assert e.value.status == dg.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.equal(dC.cpu(), C)
