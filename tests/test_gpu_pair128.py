"""CTA pair for small M (tuning variant 8): one tcgen05.mma of M = 128 over a
pair of CTAs, each loading 64 rows of A and half of a 128 x bn tile's B.

The cases cover every kind, the three tile widths, one and two row bands,
M below 64 (the second CTA's rows all outside C), ragged N (the last tile's
second half past N), an odd number of K blocks (a stage with one block), and
beta on and off.  Results must match the oracle within the path's tolerance.
"""
import numpy as np
import pytest
import torch

from tests import parity

pytestmark = pytest.mark.gpu

CASES = [
    ("f16_tn", (127, 12288, 4096), 256),  # the skinny workload
    ("f16_tn", (127, 12288, 4096), 192),
    ("f16_tn", (127, 8192, 4096), 128),   # 64 tiles
    ("f16_tn", (100, 1000, 2048), 192),   # ragged N
    ("f16_tn", (40, 2048, 1000), 256),    # M < 64: the second CTA stores nothing
    ("f16_tn", (200, 2000, 1000), 128),   # two row bands
    ("f16_tn", (128, 520, 200), 256),     # K = 200: four K blocks, the last one partial
    ("bf16_tn", (127, 4096, 1088), 192),  # 17 K blocks: a last stage of one block
    ("tf32", (127, 4096, 1000), 256),
    ("tf32", (100, 1000, 520), 192),
    ("f16_nn", (127, 4096, 1000), 256),
    ("bf16_nn", (100, 1088, 520), 128),
]


def _ids(c):
    return "%s-%dx%dx%d-bn%d" % (c[0], *c[1], c[2])


@pytest.mark.parametrize("path,shape,bn", CASES, ids=[_ids(c) for c in CASES])
def test_pair128_matches_oracle(path, shape, bn):
    import dense_gemm_09_gb300 as dg
    M, N, K = shape
    A, B, C = parity.host_operands(path, M, N, K, seed=M + 5 * N + K + bn)
    for alpha, beta in ((1.0, 0.0), (0.75, -0.5)):
        dg.tune_next(dg.TUNE_PAIR128, bn, 1)
        got, _, _ = parity.run(path, A, B, C, alpha, beta)
        assert "_pair_128x%dx" % bn in dg.last_kernel(), dg.last_kernel()
        assert dg.device_status() == dg.OK
        assert parity.worst_ratio(path, got, A, B, C, alpha, beta) <= 1.0


@pytest.mark.parametrize("path", ["f16_tn", "tf32", "bf16_nn"])
def test_pair128_integers_bit_exact(path):
    import dense_gemm_09_gb300 as dg
    M, N, K = 120, 1024, 1024
    A, B, C = parity.host_operands(path, M, N, K, seed=17, dist="int")
    dg.tune_next(dg.TUNE_PAIR128, 256, 1)
    got, _, _ = parity.run(path, A, B, C, 1.0, 1.0)
    assert "_pair_128x256x" in dg.last_kernel(), dg.last_kernel()
    ref, _ = parity.reference(path, A, B, C, 1.0, 1.0)
    assert np.array_equal(got.double().numpy(), ref)


@pytest.mark.parametrize("path,shape,bn", [("f16_tn", (127, 65536, 256), 256),   # 256 tiles: beyond one wave
                                           ("f16_nn", (127, 4096, 512), 192)])   # 96 columns: not whole B boxes
def test_pair128_request_falls_back(path, shape, bn):
    import dense_gemm_09_gb300 as dg
    M, N, K = shape
    A, B, C = parity.host_operands(path, M, N, K, seed=3)
    dg.tune_next(dg.TUNE_PAIR128, bn, 1)
    got, _, _ = parity.run(path, A, B, C, 1.0, 0.0)
    assert "_pair_128x" not in dg.last_kernel(), dg.last_kernel()
    assert parity.worst_ratio(path, got, A, B, C, 1.0, 0.0) <= 1.0


def test_pair128_is_deterministic():
    import dense_gemm_09_gb300 as dg
    A, B, C = parity.host_operands("f16_tn", 127, 12288, 4096, seed=5)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    outs = []
    for _ in range(3):
        o = dC.clone()
        dg.tune_next(dg.TUNE_PAIR128, 256, 1)
        parity.fn("f16_tn")(dA, dB, o, 1.0, 1.0)
        outs.append(o)
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_pair128_stall_times_out_cleanly():
    """A stalled launch: the MMA's wait runs out, the producers and epilogues
    give up within their limits, the status reports the time-out, and the
    next launch is exact."""
    import dense_gemm_09_gb300 as dg
    A, B, C = parity.host_operands("f16_tn", 127, 4096, 1024, seed=4)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    torch.cuda.synchronize()
    assert dg.device_status(clear=True) == dg.OK
    out = dC.clone()
    dg.tune_next(dg.TUNE_PAIR128, 256, 1)
    dg.test_inject_stall(20_000_000)  # 20 ms
    parity.fn("f16_tn")(dA, dB, out, 1.0, 0.0)
    st = dg.device_status(clear=True)
    assert "_pair_128x" in dg.last_kernel()
    assert st == dg.ERR_TIMEOUT, dg.status_string(st)
    dg.tune_next(dg.TUNE_PAIR128, 256, 1)
    got, _, _ = parity.run("f16_tn", A, B, C, 1.0, 0.0)
    assert dg.device_status(clear=True) == dg.OK
    assert parity.worst_ratio("f16_tn", got, A, B, C, 1.0, 0.0) <= 1.0


@pytest.mark.parametrize("path", ["f16_tn", "f16_nn", "bf16_tn", "bf16_nn", "tf32"])
def test_automatic_choice_for_the_skinny_workload(path):
    """One band of rows and 48 tiles of 128 x 256: the 16-bit kinds take the
    small-M pair (measured fastest there), TF32 does not (it measured slower)."""
    import ctypes
    import dense_gemm_09_gb300 as dg
    kind = {"f16_tn": 0, "tf32": 1, "bf16_tn": 2, "f16_nn": 3, "bf16_nn": 4}[path]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out = [ctypes.c_int() for _ in range(3)]
    assert dg.lib().dgemm_test_choose_config(kind, 127, 12288, 4096, sms, *(ctypes.byref(o) for o in out)) == dg.OK
    v, bn, sp = (o.value for o in out)
    if path == "tf32":
        assert v != dg.TUNE_PAIR128, (v, bn, sp)
    else:
        assert (v, bn) == (dg.TUNE_PAIR128, 256), (v, bn, sp)
