"""Failure detection on the GPU without a fault: the bounded mbarrier waits.

A test-only hook makes the next launch of a kernel with bounded waits (the
tensor-core kernels and the TMA-fed FP32 SIMT kernel) first wait on a
barrier nothing arrives at, so that wait (and then every other role's) runs
out after a short limit.  The kernel must end by itself, record
DGEMM_ERR_TIMEOUT in the device status word, release its resources, and leave
the context usable: the next ordinary call is correct."""
import time

import pytest
import torch

from tests import parity

pytestmark = pytest.mark.gpu

# (path, shape, pitch padding, tile configuration forced through the tuning
# hook or None for the automatic choice, expected variant name fragment)
CASES = [
    ("f16_tn", (256, 512, 256), (0, 0, 0), "pair", "_pair_"),             # CTA-pair kernel
    ("tf32", (256, 512, 256), (0, 0, 0), "pair", "_pair_"),
    ("f16_tn", (128, 512, 256), (0, 0, 0), "single", "_128x256x64_tma"),  # single-CTA kernel
    ("tf32", (100, 260, 36), (1, 0, 0), None, "_cpasync"),    # cp.async producer (unaligned TF32)
    ("f16_tn", (100, 260, 36), (1, 0, 0), None, "_ldst"),     # register-path producer (unaligned FP16)
    ("f16_tn", (100, 1000, 2048), (0, 0, 0), None, "_splitk"),  # split-K cluster kernel
    ("f32", (2048, 2560, 256), (0, 0, 0), None, "sgemm_simt_tma_"),  # TMA-fed FP32 SIMT kernel
]


@pytest.mark.parametrize("path,shape,pad,force,variant", CASES,
                         ids=[c[4].strip("_") + "-" + c[0] for c in CASES])
def test_stalled_launch_times_out_cleanly(path, shape, pad, force, variant):
    import dense_gemm_09_gb300 as dg
    M, N, K = shape
    A, B, C = parity.host_operands(path, M, N, K, seed=3)
    dA, _ = parity.to_device_padded(A, pad[0])
    dB, _ = parity.to_device_padded(B, pad[1])
    dC = C.cuda()
    torch.cuda.synchronize()
    assert dg.device_status(clear=True) == dg.OK
    fn = {"tf32": dg.gemm_tf32, "f16_tn": dg.gemm_f16_tn, "f32": dg.gemm_f32}[path]

    if force == "pair":
        dg.tune_next(dg.TUNE_PAIR)
    elif force == "single":
        dg.tune_next(dg.TUNE_SINGLE, 256)
    dg.test_inject_stall(20_000_000)  # 20 ms
    t0 = time.monotonic()
    fn(dA, dB, dC, 1.0, 0.0)
    st = dg.device_status(clear=True)  # synchronises (and clears before any assert below)
    assert variant in dg.last_kernel()
    elapsed = time.monotonic() - t0
    assert st == dg.ERR_TIMEOUT, dg.status_string(st)
    assert elapsed < 10.0

    # the context is usable and the next call (no injection) is correct
    fn(dA, dB, dC, 1.5, 0.0)
    torch.cuda.synchronize()
    assert dg.device_status(clear=True) == dg.OK
    assert parity.worst_ratio(path, dC.cpu(), A, B, C, 1.5, 0.0) <= 1.0


def test_injection_is_one_shot():
    import dense_gemm_09_gb300 as dg
    A, B, C = parity.host_operands("f16_tn", 256, 256, 128, seed=4)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    dg.test_inject_stall(10_000_000)
    dg.gemm_f16_tn(dA, dB, dC, 1.0, 0.0)
    assert dg.device_status(clear=True) == dg.ERR_TIMEOUT
    for _ in range(3):
        dg.gemm_f16_tn(dA, dB, dC, 1.0, 0.0)
    assert dg.device_status(clear=True) == dg.OK
    assert parity.worst_ratio("f16_tn", dC.cpu(), A, B, C, 1.0, 0.0) <= 1.0
