"""Stream-K tail of the CTA-pair kernels.

When the output tiles outnumber the CTA pairs and do not divide evenly, the
first P + (T mod P) tiles are cut along K into one contiguous range per pair.
The pair that continues a cut tile starts from the partial accumulator the
previous pair left in the library's workspace, so its MMAs run in the same
order as for an uncut tile: the results must equal the round-robin schedule
bit for bit, and the oracle within the path's tolerance.
"""
import pytest
import torch

from tests import parity

pytestmark = pytest.mark.gpu

# (path, M, N, K): tile counts on 76 pairs -- 10 x 9 = 90 wide tiles (every
# tile cut, ragged edges); 16 x 10 = 160 wide tiles (84 cut, 76 whole);
# 9 x 9 = 81 tiles of 256 x 256
CASES = [
    ("f16_tn", 2500, 4500, 1000),
    ("tf32", 2500, 4500, 1000),
    ("bf16_tn", 4096, 5120, 512),
    ("f16_nn", 4096, 5120, 520),
    ("tf32", 4096, 5120, 260),
]


def _run(path, dA, dB, C0, alpha, beta, variant, sk):
    import dense_gemm_09_gb300 as dg
    out = C0.clone()
    dg.tune_next(variant, 256, sk)
    parity.fn(path)(dA, dB, out, alpha, beta)
    torch.cuda.synchronize()
    return out, dg.last_kernel()


@pytest.mark.parametrize("path,M,N,K", CASES, ids=["%s-%dx%dx%d" % c for c in CASES])
@pytest.mark.parametrize("wide", [True, False], ids=["256x512", "256x256"])
def test_stream_k_equals_round_robin_bitwise(path, M, N, K, wide):
    import dense_gemm_09_gb300 as dg
    if not wide:
        M, N = min(M, 2304), min(N, 2304)  # 9 x 9 tiles of 256 x 256
    A, B, C = parity.host_operands(path, M, N, K, seed=M + N + K)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    variant = dg.TUNE_PAIR_WIDE if wide else dg.TUNE_PAIR
    whole, name0 = _run(path, dA, dB, dC, 1.25, -0.5, variant, dg.SK_OFF)
    cut, name1 = _run(path, dA, dB, dC, 1.25, -0.5, variant, dg.SK_ON)
    assert "_sk_" not in name0 and "_sk_" in name1, (name0, name1)
    assert dg.device_status() == dg.OK
    assert torch.equal(whole, cut)


@pytest.mark.parametrize("path", ["f16_tn", "bf16_tn"])
@pytest.mark.parametrize("wide", [True, False], ids=["256x512", "256x256"])
def test_finer_ring_matches_oracle_and_coarse_ring(path, wide):
    """The finer stage ring (32-deep K stages under the 64-byte swizzle) runs
    the same MMAs in the same K order as the ordinary ring: results agree
    bit for bit, whole tiles and stream-K alike, and with the oracle."""
    import dense_gemm_09_gb300 as dg
    M, N, K = (2500, 4500, 1000) if wide else (2304, 2304, 1000)
    A, B, C = parity.host_operands(path, M, N, K, seed=M + K)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    coarse = dg.TUNE_PAIR_WIDE if wide else dg.TUNE_PAIR
    fine = dg.TUNE_PAIR_WIDE_FINE if wide else dg.TUNE_PAIR_FINE
    want, _ = _run(path, dA, dB, dC, 0.75, 0.5, coarse, dg.SK_OFF)
    for sk in (dg.SK_OFF, dg.SK_ON):
        got, name = _run(path, dA, dB, dC, 0.75, 0.5, fine, sk)
        assert ("x32_sk_tma" if sk == dg.SK_ON else "x32_tma") in name, name
        assert dg.device_status() == dg.OK
        assert torch.equal(got, want)
    assert parity.worst_ratio(path, got.cpu(), A, B, C, 0.75, 0.5) <= 1.0


def test_finer_ring_request_falls_back_for_n_major_kinds():
    import dense_gemm_09_gb300 as dg
    A, B, C = parity.host_operands("tf32", 600, 1100, 520, seed=3)
    got, name = _run("tf32", A.cuda(), B.cuda(), C.cuda(), 1.0, 0.0, dg.TUNE_PAIR_FINE, dg.SK_OFF)
    assert "_pair_256x256x32_tma" in name, name  # the ordinary ring (TF32's stages are 32 deep already)
    assert parity.worst_ratio("tf32", got.cpu(), A, B, C, 1.0, 0.0) <= 1.0


@pytest.mark.parametrize("path", ["f16_tn", "tf32"])
def test_stream_k_matches_oracle(path):
    import dense_gemm_09_gb300 as dg
    M, N, K = 2500, 4500, 1000
    A, B, C = parity.host_operands(path, M, N, K, seed=11)
    dg.tune_next(dg.TUNE_PAIR_WIDE, 256, dg.SK_ON)
    got, _, _ = parity.run(path, A, B, C, 0.75, 0.5)
    assert "_sk_" in dg.last_kernel()
    assert dg.device_status() == dg.OK
    assert parity.worst_ratio(path, got, A, B, C, 0.75, 0.5) <= 1.0


@pytest.mark.parametrize("path,shape", [("f16_tn", (4096, 4096, 4096)), ("tf32", (2560, 4096, 2048)),
                                        ("tf32", (12288, 12288, 4096))])
def test_automatic_choice_takes_stream_k(path, shape):
    """256 / 160 tiles of 256 x 256 and 1152 of 256 x 512 on 76 pairs: the
    automatic choice cuts the tail, and matches the uncut schedule of the same
    tile shape exactly."""
    import dense_gemm_09_gb300 as dg
    M, N, K = shape
    A, B, C = parity.host_operands(path, M, N, K, seed=5)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    auto = dC.clone()
    parity.fn(path)(dA, dB, auto, 1.0, 0.0)
    torch.cuda.synchronize()
    name = dg.last_kernel()
    assert "_pair_" in name and "_sk_" in name, name
    variant = dg.TUNE_PAIR_WIDE if "_pair_256x512x" in name else dg.TUNE_PAIR
    whole, _ = _run(path, dA, dB, dC, 1.0, 0.0, variant, dg.SK_OFF)
    assert torch.equal(auto, whole)
    assert parity.sampled_check(path, auto, A, B, C, 1.0, 0.0, n_samples=2048) <= 1.0


def test_stream_k_is_not_captured_in_graphs():
    """Under stream capture the round-robin schedule runs (the graph would
    otherwise hold the shared workspace); replays equal the eager result."""
    import dense_gemm_09_gb300 as dg
    path, (M, N, K) = "f16_tn", (2500, 4500, 1000)
    A, B, C = parity.host_operands(path, M, N, K, seed=2)
    dA, dB = A.cuda(), B.cuda()
    eager = C.cuda()
    dg.tune_next(dg.TUNE_PAIR_WIDE, 256, dg.SK_ON)
    parity.fn(path)(dA, dB, eager, 1.0, 0.0)
    torch.cuda.synchronize()
    assert "_sk_" in dg.last_kernel()
    out = torch.empty_like(eager)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            dg.tune_next(dg.TUNE_PAIR_WIDE, 256, dg.SK_ON)
            parity.fn(path)(dA, dB, out, 1.0, 0.0)
    assert "_sk_" not in dg.last_kernel(), dg.last_kernel()
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)


def test_stream_k_launches_on_several_streams():
    """Stream-K launches from different streams share one workspace; they
    are ordered one after another and each result is exact."""
    import dense_gemm_09_gb300 as dg
    path, (M, N, K) = "tf32", (2500, 4500, 1000)
    A, B, C = parity.host_operands(path, M, N, K, seed=9)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    want, _ = _run(path, dA, dB, dC, 1.0, 1.0, dg.TUNE_PAIR_WIDE, dg.SK_OFF)
    streams = [torch.cuda.Stream() for _ in range(4)]
    outs = []
    for rep in range(3):
        for s in streams:
            with torch.cuda.stream(s):
                o = dC.clone()
                dg.tune_next(dg.TUNE_PAIR_WIDE, 256, dg.SK_ON)
                parity.fn(path)(dA, dB, o, 1.0, 1.0)
                outs.append(o)
    torch.cuda.synchronize()
    assert dg.device_status() == dg.OK
    for o in outs:
        assert torch.equal(o, want)


def test_stream_k_on_two_streams_matches_oracle():
    """Two different stream-K problems (TF32 and FP16 TN) issued back to back
    on two independent streams: the library orders them through its event
    (they share the workspace), and each result agrees with the oracle."""
    import dense_gemm_09_gb300 as dg
    probs = []
    for path, seed in (("tf32", 21), ("f16_tn", 22)):
        M, N, K = 2500, 4500, 1000
        A, B, C = parity.host_operands(path, M, N, K, seed=seed)
        probs.append((path, A, B, C, A.cuda(), B.cuda(), C.cuda()))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    names = []
    for (path, _, _, _, dA, dB, dC), s in zip(probs, streams):
        with torch.cuda.stream(s):
            dg.tune_next(dg.TUNE_PAIR_WIDE, 256, dg.SK_ON)
            parity.fn(path)(dA, dB, dC, 0.75, 0.5)
            names.append(dg.last_kernel())
    torch.cuda.synchronize()
    assert all("_sk_" in n for n in names), names
    assert dg.device_status() == dg.OK
    for path, A, B, C, _, _, dC in probs:
        assert parity.worst_ratio(path, dC.cpu(), A, B, C, 0.75, 0.5) <= 1.0


def test_stream_k_stall_times_out_cleanly():
    """A stalled stream-K launch: the MMA waits run out, the pairs waiting for
    a partial give up within their own limit, and the next launch (a new
    generation of flags) is exact."""
    import dense_gemm_09_gb300 as dg
    path, (M, N, K) = "f16_tn", (2500, 4500, 1000)
    A, B, C = parity.host_operands(path, M, N, K, seed=4)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    torch.cuda.synchronize()
    assert dg.device_status(clear=True) == dg.OK
    out = dC.clone()
    dg.tune_next(dg.TUNE_PAIR_WIDE, 256, dg.SK_ON)
    dg.test_inject_stall(20_000_000)  # 20 ms
    parity.fn(path)(dA, dB, out, 1.0, 0.0)
    st = dg.device_status(clear=True)
    assert "_sk_" in dg.last_kernel()
    assert st == dg.ERR_TIMEOUT, dg.status_string(st)
    cut, _ = _run(path, dA, dB, dC, 1.0, 0.0, dg.TUNE_PAIR_WIDE, dg.SK_ON)
    whole, _ = _run(path, dA, dB, dC, 1.0, 0.0, dg.TUNE_PAIR_WIDE, dg.SK_OFF)
    assert dg.device_status(clear=True) == dg.OK
    assert torch.equal(cut, whole)
