"""gemm_tf32_noalloc: the TF32 GEMM for callers that cannot allocate device
memory (for example code inside a framework whose memory pool owns the whole
device, or a loop that must not allocate), who therefore cannot hand
gemm_tf32_ws a workspace.  The copies of operands that TMA cannot load go to
a fixed scratch array inside the library instead.

Checked on the GPU through the C ABI, on two calls in a row (the second call
reuses the scratch the first one filled): each result is compared element by
element with the CPU oracle, within the TF32 tolerance the parity tests use,
and with gemm_tf32_ws given a workspace (the existing entry point), which
runs the same kernels on the same copies and so must agree bit for bit.  This file is collected last so that a run stopping at the first
failure has run every other test; it also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

from tests import parity

pytestmark = pytest.mark.gpu


def _unaligned_operands(M, N, K, seed):
    # tight pitches with K and N not multiples of 4: neither A nor B can be
    # loaded by TMA as stored, so both go through the scratch
    A, B, C = parity.host_operands("tf32", M, N, K, seed=seed)
    return A, B, C, A.cuda(), B.cuda()


def _noalloc(L, dA, dB, dC, alpha, beta):
    M, K = dA.shape
    N = dB.shape[1]
    return L.gemm_tf32_noalloc(M, N, K, ctypes.c_float(alpha), dA.data_ptr(), dA.stride(0),
                               dB.data_ptr(), dB.stride(0), ctypes.c_float(beta), dC.data_ptr(),
                               dC.stride(0), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_oracle_and_workspace_entry_on_two_calls():
    import dense_gemm_09_gb300 as dg
    L = dg.lib()
    cases = [((1000, 1501, 1001), 21, 1.5, -0.25),   # both operands copied
             ((777, 2049, 515), 22, 0.75, 0.5)]      # different shape: the scratch is reused
    for (M, N, K), seed, alpha, beta in cases:
        A, B, C, dA, dB = _unaligned_operands(M, N, K, seed)
        need = dg.tf32_workspace_bytes(dA, dB)
        assert 0 < need <= dg.NOALLOC_SCRATCH_BYTES
        got = C.cuda()
        assert _noalloc(L, dA, dB, got, alpha, beta) == dg.OK
        assert dg.last_kernel().endswith("_tma"), dg.last_kernel()
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        want = C.cuda()
        dg.gemm_tf32_ws(dA, dB, want, alpha, beta, workspace=ws)
        torch.cuda.synchronize()
        assert dg.device_status() == dg.OK
        # the oracle decides: |got - ref| <= tol*(|A||B|) + tol*|beta*c| per element
        assert parity.worst_ratio("tf32", got.cpu(), A, B, C, alpha, beta) <= 1.0
        # same kernels on the same copied values: the results agree exactly
        assert torch.equal(got, want)


def test_noalloc_refuses_operands_beyond_the_scratch():
    import dense_gemm_09_gb300 as dg
    L = dg.lib()
    # A alone: 4097 rows x 4100 floats = 67.2 MB > 64 MiB
    M, N, K = 4097, 64, 4097
    dA = torch.ones((M, K), device="cuda")
    dB = torch.ones((K, N), device="cuda")
    C = torch.full((M, N), 7.0, device="cuda")
    assert dg.tf32_workspace_bytes(dA, dB) > dg.NOALLOC_SCRATCH_BYTES
    assert _noalloc(L, dA, dB, C, 1.0, 0.0) == dg.ERR_INVALID_ARG
    with pytest.raises(dg.DgemmError, match="fixed scratch"):
        dg.gemm_tf32_noalloc(dA, dB, C)
    torch.cuda.synchronize()
    assert bool((C == 7.0).all())  # nothing was launched


def test_noalloc_aligned_operands_need_no_scratch():
    import dense_gemm_09_gb300 as dg
    L = dg.lib()
    M, N, K = 512, 768, 1024
    A, B, C = parity.host_operands("tf32", M, N, K, seed=23)
    dA, dB = A.cuda(), B.cuda()
    assert dg.tf32_workspace_bytes(dA, dB) == 0
    got = C.cuda()
    assert _noalloc(L, dA, dB, got, 1.0, 0.5) == dg.OK
    want = C.cuda()
    dg.gemm_tf32(dA, dB, want, 1.0, 0.5)
    torch.cuda.synchronize()
    assert parity.worst_ratio("tf32", got.cpu(), A, B, C, 1.0, 0.5) <= 1.0
    assert torch.equal(got, want)
