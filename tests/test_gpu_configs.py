"""The workload configurations at full size, on the GPU, against the oracle.

Each configuration runs through the C ABI with its seeded operands; the
result is compared with the oracle in full where the oracle finishes in
seconds (M*N*K <= 2^37 on the machine's host cores) and otherwise on 4096
seeded entries plus full rows and columns at tile boundaries.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from tests import parity

pytestmark = pytest.mark.gpu

CASES = [
    # (workload, path, full check)
    ("f32_256", "f32", True),
    ("f32_256", "tf32", True),
    ("f32_4092", "f32", True),
    ("f32_4092", "tf32", True),
    ("f32_8192x8192x4096", "f32", False),
    ("f32_8192x8192x4096", "tf32", False),
    ("f32_8191x8193x4095", "f32", False),
    ("f32_8191x8193x4095", "tf32", False),
    ("f16_tn_2048", "f16_tn", True),
    ("f16_tn_4096", "f16_tn", True),
    ("f16_tn_8192", "f16_tn", False),
    ("f16_tn_12288", "f16_tn", False),
    ("f16_tn_16384", "f16_tn", False),
    ("f16_tn_8192x8192x4096", "f16_tn", False),
    ("f16_tn_127x12288x4096", "f16_tn", True),
]


@pytest.mark.parametrize("name,path,full", CASES, ids=[c[0] + "-" + c[1] for c in CASES])
def test_config(name, path, full):
    import dense_gemm_09_gb300 as dg
    w = si.WORKLOADS[name]
    A, B, C = si.make(w)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    fn = {"f32": dg.gemm_f32, "tf32": dg.gemm_tf32, "f16_tn": dg.gemm_f16_tn}[path]
    fn(dA, dB, dC, w.alpha, w.beta)
    torch.cuda.synchronize()
    assert dg.device_status() == dg.OK
    if full:
        worst = parity.worst_ratio(path, dC.cpu(), A, B, C, w.alpha, w.beta)
    else:
        worst = parity.sampled_check(path, dC, A, B, C, w.alpha, w.beta)
    assert worst <= 1.0, worst
    assert torch.isfinite(dC).all()


# The layout / type variants at a full square size: FP16 NN and BF16 TN / NN,
# seeded uniform operands (rounded to the 16-bit type), checked in full.
@pytest.mark.parametrize("path", ["f16_nn", "bf16_tn", "bf16_nn"])
def test_variant_4096_cube_full(path):
    import dense_gemm_09_gb300 as dg
    A, B, C = parity.host_operands(path, 4096, 4096, 4096, seed=17)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    parity.fn(path)(dA, dB, dC, 1.5, -0.25)
    torch.cuda.synchronize()
    assert dg.device_status() == dg.OK
    assert "_pair_" in dg.last_kernel()
    assert parity.worst_ratio(path, dC.cpu(), A, B, C, 1.5, -0.25) <= 1.0
