"""Parity of the CUDA paths (through the C ABI) with the CPU oracle.

Small and ragged shapes are compared in full, element by element, against
the acceptance rule |C_gpu - ref| <= tol*(|A||B|)_ij + tol*|beta*c_ij| with
tol = 1e-6*sqrt(K) (FP32), 2e-3 (TF32), 1e-3 (FP16 -> FP32).  Small-integer
operands make every path exact, so those cases are compared bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import seeded_inputs as si
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import dense_gemm_09_gb300 as dg
    dg.lib()
    dg.device_status(clear=True)
    yield dg
    assert dg.device_status(clear=True) == dg.OK


# Shapes: tiny, tile-exact, ragged in every dimension, several tiles, and a
# tile count above the SM count (persistent CTAs take several tiles).
SHAPES = {
    "f32": [(1, 1, 1), (5, 7, 3), (17, 9, 33), (31, 33, 32), (128, 128, 16), (129, 127, 17),
            (255, 257, 300), (300, 520, 1000), (1, 300, 700), (700, 1, 300), (64, 1000, 5)],
    # TF32 / FP16: 16-byte multiples of the row pitch take the TMA producer,
    # the others (odd K for A, odd N for TF32's B) the register-path producer
    "tf32": [(1, 4, 4), (5, 8, 12), (17, 12, 36), (128, 256, 32), (129, 260, 36), (255, 516, 300),
             (300, 520, 1000), (1, 300, 704), (700, 4, 300), (64, 1000, 8),
             (1, 1, 1), (5, 7, 3), (17, 9, 33), (129, 127, 17), (255, 257, 301)],
    "f16_tn": [(1, 1, 8), (5, 7, 16), (17, 9, 40), (128, 256, 64), (129, 257, 72), (255, 513, 304),
               (300, 520, 1000), (1, 300, 704), (700, 1, 304), (64, 1000, 8),
               (1, 1, 1), (5, 7, 3), (17, 9, 33), (129, 127, 17), (255, 257, 301)],
}
# The other 16-bit paths (FP16 NN, BF16 TN / NN) take the FP16 TN shape list:
# NN pitches of N elements are TMA-capable when N is a multiple of 8.
for _p in ("f16_nn", "bf16_tn", "bf16_nn"):
    SHAPES[_p] = SHAPES["f16_tn"]


@pytest.mark.parametrize("path,shape", [(p, s) for p in parity.PATHS for s in SHAPES[p]])
def test_random_shapes_full(path, shape):
    M, N, K = shape
    A, B, C = parity.host_operands(path, M, N, K, seed=M + 7 * N + 13 * K)
    got, _, _ = parity.run(path, A, B, C, 1.5, -0.25)
    assert parity.worst_ratio(path, got, A, B, C, 1.5, -0.25) <= 1.0


@pytest.mark.parametrize("path", parity.PATHS)
def test_beta_zero_alpha_one(path):
    M, N, K = 200, 264, 136
    A, B, C = parity.host_operands(path, M, N, K, seed=3)
    got, _, _ = parity.run(path, A, B, C, 1.0, 0.0)
    assert parity.worst_ratio(path, got, A, B, C, 1.0, 0.0) <= 1.0


@pytest.mark.parametrize("path,shape", [
    ("f32", (64, 72, 300)), ("f32", (129, 257, 1000)),
    ("tf32", (64, 72, 300)), ("tf32", (129, 260, 1000)),
    ("f16_tn", (64, 72, 304)), ("f16_tn", (129, 257, 1024)),
    ("f16_nn", (64, 72, 304)), ("f16_nn", (129, 264, 1024)),
    # bfloat16 holds integers exactly up to 256: |sum| <= K + 1 must stay below
    ("bf16_tn", (64, 72, 200)), ("bf16_tn", (129, 257, 248)),
    ("bf16_nn", (64, 72, 200)), ("bf16_nn", (129, 264, 248))])
def test_small_integers_bit_exact(path, shape):
    # every partial sum is an integer below 2^24: any summation order is exact
    M, N, K = shape
    A, B, C = parity.host_operands(path, M, N, K, seed=11, dist="int")
    beta = 2.0 if path in ("f32", "tf32") else 1.0
    got, _, _ = parity.run(path, A, B, C, 1.0, beta)
    ref, _ = parity.reference(path, A, B, C, 1.0, beta)
    assert np.array_equal(got.double().numpy(), ref)


@pytest.mark.parametrize("path", parity.PATHS)
def test_identity_and_permutation_exact(path):
    M = 136
    N = 264
    g = si.generator(5)
    dt = parity.dtype(path)
    perm = torch.randperm(M, generator=g)
    P = torch.zeros((M, M), dtype=dt)
    P[torch.arange(M), perm] = 1
    Bl = si.uniform((M, N), g).to(dt)          # logical B (K x N)
    B = Bl.T.contiguous() if parity.is_tn(path) else Bl
    C = torch.zeros((M, N), dtype=dt)
    got, _, _ = parity.run(path, P, B, C, 1.0, 0.0)
    want = Bl[perm]
    if path == "tf32":
        # the product reads B through TF32: compare with the oracle's exact values
        ref, _ = parity.reference(path, P, B, C, 1.0, 0.0)
        assert np.array_equal(got.double().numpy(), ref)
    else:
        assert torch.equal(got, want)


@pytest.mark.parametrize("path", parity.PATHS)
def test_alpha_zero_does_not_read_a_b(path):
    M, N, K = 70, 136, 64
    A, B, C = parity.host_operands(path, M, N, K, seed=2)
    A = torch.full_like(A, float("nan"))
    B = torch.full_like(B, float("nan"))
    got, _, _ = parity.run(path, A, B, C, 0.0, 0.5)
    want = (C.double() * 0.5)
    assert torch.equal(got.double(), want.to(got.dtype).double())


@pytest.mark.parametrize("path", parity.PATHS)
def test_beta_zero_does_not_read_c(path):
    M, N, K = 70, 136, 64
    A, B, C = parity.host_operands(path, M, N, K, seed=4)
    Cnan = torch.full_like(C, float("nan"))
    got, _, _ = parity.run(path, A, B, Cnan, 1.0, 0.0)
    assert torch.isfinite(got).all()
    assert parity.worst_ratio(path, got, A, B, C, 1.0, 0.0) <= 1.0


@pytest.mark.parametrize("path", parity.PATHS)
def test_k_zero_scales_c(path):
    M, N = 33, 40
    _, _, C = parity.host_operands(path, M, N, 8, seed=6)
    A = torch.zeros((M, 0), dtype=C.dtype)
    B = torch.zeros((N, 0) if parity.is_tn(path) else (0, N), dtype=C.dtype)
    got, _, _ = parity.run(path, A, B, C, 1.0, -2.0)
    assert torch.equal(got, (C.double() * -2.0).to(C.dtype))
    got, _, _ = parity.run(path, A, B, C, 1.0, 0.0)
    assert torch.equal(got, torch.zeros_like(C))


@pytest.mark.parametrize("path", parity.PATHS)
def test_empty_m_or_n_is_a_no_op(path):
    dt = parity.dtype(path)
    fn = parity.fn(path)
    for M, N in ((0, 16), (16, 0)):
        A = torch.ones((M, 8), dtype=dt, device="cuda")
        B = torch.ones((N, 8) if parity.is_tn(path) else (8, N), dtype=dt, device="cuda")
        C = torch.ones((M, N), dtype=dt, device="cuda")
        fn(A, B, C, 1.0, 1.0)
    torch.cuda.synchronize()


@pytest.mark.parametrize("path", parity.PATHS)
def test_padded_leading_dims_and_canaries(path):
    # C lives in a wider buffer filled with NaN; only the M x N entries change
    M, N, K = 150, 264, 200
    A, B, C = parity.host_operands(path, M, N, K, seed=8)
    pad = (8, 8, 32)  # keeps 16-byte row pitches for every path
    got, dC, cbuf = parity.run(path, A, B, C, 1.0, 0.5, pad=pad)
    assert parity.worst_ratio(path, got, A, B, C, 1.0, 0.5) <= 1.0
    ld = N + pad[2]
    rows = cbuf[:M * ld].view(M, ld)
    assert torch.isnan(rows[:, N:]).all()          # padding columns untouched
    assert torch.isnan(cbuf[M * ld:]).all()        # rows past M untouched


def test_f32_unaligned_leading_dims():
    # odd pitches and a base pointer off a 16-byte boundary: scalar-load path
    M, N, K = 131, 133, 137
    A, B, C = parity.host_operands("f32", M, N, K, seed=9)
    got, _, _ = parity.run("f32", A, B, C, 1.5, -0.25, pad=(1, 3, 1), offset=(1, 2, 3))
    assert parity.worst_ratio("f32", got, A, B, C, 1.5, -0.25) <= 1.0


@pytest.mark.parametrize("path", ["tf32", "f16_tn"])
def test_many_tiles_per_cta(path):
    # more tiles than SMs: each persistent CTA runs several tiles and both
    # TMEM accumulators
    M, N, K = 2048, 4096, 192
    A, B, C = parity.host_operands(path, M, N, K, seed=10)
    got, dC, _ = parity.run(path, A, B, C, 1.0, 0.5)
    assert parity.sampled_check(path, dC, A, B, C, 1.0, 0.5) <= 1.0


def test_stream_argument_is_honoured():
    import dense_gemm_09_gb300 as dg
    s = torch.cuda.Stream()
    A, B, C = parity.host_operands("f32", 256, 256, 256, seed=12)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        dg.gemm_f32(dA, dB, dC, 1.0, 1.0, stream=s)
    s.synchronize()
    assert parity.worst_ratio("f32", dC.cpu(), A, B, C, 1.0, 1.0) <= 1.0


def test_tf32_operand_rounding_is_truncation():
    # Crafted operands decide how FP32 values are reduced to TF32 inside the
    # multiplier: 1+2^-11 is a tie (nearest-away gives 1+2^-10), 1+2^-11+2^-13
    # is above the tie (any nearest mode gives 1+2^-10).  Truncation keeps 1.
    import dense_gemm_09_gb300 as dg
    xs = [1 + 2**-11, 1 + 2**-11 + 2**-13, 1 + 2**-12, -(1 + 2**-11), 1 + 3 * 2**-11, 3.0]
    K = 8
    A = torch.zeros((len(xs), K))
    A[:, 0] = torch.tensor(xs)
    B = torch.zeros((K, 8))
    B[0, :] = 1.0
    C = torch.zeros((len(xs), 8))
    got, _, _ = parity.run("tf32", A, B, C, 1.0, 0.0)
    want = [1.0, 1.0, 1.0, -1.0, 1 + 2**-10, 3.0]
    assert got[:, 0].tolist() == want
    ref, _ = parity.reference("tf32", A, B, C, 1.0, 0.0)
    assert np.array_equal(got.numpy().astype(np.float64), ref)


@pytest.mark.parametrize("path", parity.TC_PATHS)
@pytest.mark.parametrize("shape,pad,offset", [
    ((131, 133, 137), (1, 3, 1), (1, 2, 3)),      # odd pitches, misaligned bases
    ((300, 520, 256), (1, 0, 0), (0, 0, 0)),      # only A's pitch is odd
    ((300, 520, 256), (0, 1, 0), (0, 0, 0)),      # only B's pitch is odd
    ((300, 520, 256), (0, 0, 0), (2, 0, 0)),      # only A's base is off 16 bytes
    ((700, 1030, 515), (3, 5, 7), (1, 1, 1)),     # several tiles per CTA
])
def test_tensor_paths_register_producer(path, shape, pad, offset):
    import dense_gemm_09_gb300 as dg
    M, N, K = shape
    A, B, C = parity.host_operands(path, M, N, K, seed=M + N + K)
    got, _, _ = parity.run(path, A, B, C, 1.5, -0.25, pad=pad, offset=offset)
    # 16-bit: loads through registers; TF32: 4-byte cp.async copies
    assert dg.last_kernel().endswith("_cpasync" if path == "tf32" else "_ldst")
    assert parity.worst_ratio(path, got, A, B, C, 1.5, -0.25) <= 1.0


@pytest.mark.parametrize("path", parity.TC_PATHS)
def test_register_producer_integers_bit_exact(path):
    M, N, K = 257, 300, (203 if path.startswith("bf16") else 259)
    A, B, C = parity.host_operands(path, M, N, K, seed=21, dist="int")
    got, _, _ = parity.run(path, A, B, C, 1.0, 1.0)
    ref, _ = parity.reference(path, A, B, C, 1.0, 1.0)
    assert np.array_equal(got.double().numpy(), ref)


@pytest.mark.parametrize("path", parity.PATHS)
def test_kernel_variant_names(path):
    import dense_gemm_09_gb300 as dg
    A, B, C = parity.host_operands(path, 256, 256, 256, seed=1)
    parity.run(path, A, B, C, 1.0, 0.0)
    want = "sgemm_simt" if path == "f32" else "umma_" + path
    assert dg.last_kernel().startswith(want)
    if path != "f32":
        # more than one wave of 128 x 256 tiles with M > 128: the CTA pair
        A, B, C = parity.host_operands(path, 2560, 2048, 64, seed=1)
        got, _, _ = parity.run(path, A, B, C, 1.0, 0.0)
        assert dg.last_kernel().endswith("_tma") and "_pair_" in dg.last_kernel()
        assert parity.worst_ratio(path, got, A, B, C, 1.0, 0.0) <= 1.0
        # half a wave to one wave of tiles: the pair too when M > 128 ...
        A, B, C = parity.host_operands(path, 2048, 2048, 64, seed=1)
        got, _, _ = parity.run(path, A, B, C, 1.0, 0.0)
        assert dg.last_kernel().endswith("_tma") and "_pair_" in dg.last_kernel()
        assert parity.worst_ratio(path, got, A, B, C, 1.0, 0.0) <= 1.0
        # ... and the single-CTA kernel, 256 wide, for a single row band
        A, B, C = parity.host_operands(path, 128, 20480, 64, seed=1)
        got, _, _ = parity.run(path, A, B, C, 1.0, 0.0)
        assert "_128x256x" in dg.last_kernel() and dg.last_kernel().endswith("_tma")
        assert parity.worst_ratio(path, got, A, B, C, 1.0, 0.0) <= 1.0


@pytest.mark.parametrize("path", parity.TC_PATHS)
@pytest.mark.parametrize("M", [129, 200, 255, 256, 257, 383, 511, 640])
def test_pair_kernel_m_tails(path, M):
    import dense_gemm_09_gb300 as dg
    # the pair tile is 256 rows: the odd CTA's rows run past M in these cases
    N, K = 520, 264
    A, B, C = parity.host_operands(path, M, N, K, seed=M)
    dg.tune_next(dg.TUNE_PAIR)  # few tiles: the automatic choice would take the single-CTA kernel
    got, _, _ = parity.run(path, A, B, C, 1.5, -0.25)
    assert "_pair_" in dg.last_kernel()
    assert parity.worst_ratio(path, got, A, B, C, 1.5, -0.25) <= 1.0


@pytest.mark.parametrize("path", ["tf32", "f16_nn", "bf16_nn"])
@pytest.mark.parametrize("N", [256, 320, 544, 576, 1000, 1024])
def test_pair_kernel_n_major_b(path, N):
    import dense_gemm_09_gb300 as dg
    # N-major B in the pair kernel: when N is a whole number of 128-byte
    # column groups (32 TF32 or 64 16-bit columns) a stage's B half is one
    # 3-D box, otherwise 128-byte 2-D boxes; N past the last pair tile's
    # first half (320, 544, 576, 1000) leaves the odd CTA's columns partly or
    # wholly outside B.
    M, K = 300, 520
    A, B, C = parity.host_operands(path, M, N, K, seed=N)
    dg.tune_next(dg.TUNE_PAIR)
    got, _, _ = parity.run(path, A, B, C, 0.75, 0.5)
    assert "_pair_" in dg.last_kernel()
    assert parity.worst_ratio(path, got, A, B, C, 0.75, 0.5) <= 1.0


@pytest.mark.parametrize("path", parity.TC_PATHS)
@pytest.mark.parametrize("shape", [(300, 520, 264), (520, 1000, 200), (1000, 768, 520), (257, 1536, 64),
                                   (129, 300, 40)])
def test_pair_wide_kernel(path, shape):
    import dense_gemm_09_gb300 as dg
    # 256 x 512 pair tiles (two N = 256 MMAs per step, one 512-column
    # accumulator, eight epilogue warps); N not a multiple of 512 leaves the
    # tile's second half partly (1000) or wholly (300, 520) outside C
    M, N, K = shape
    if path.endswith("_nn") and N % 8:
        N += 8 - N % 8  # a 16-bit NN B's pitch (N) must be a 16-byte multiple for TMA
    A, B, C = parity.host_operands(path, M, N, K, seed=3 * M + N)
    dg.tune_next(dg.TUNE_PAIR_WIDE)
    got, _, _ = parity.run(path, A, B, C, 1.25, -0.5)
    assert "_pair_256x512x" in dg.last_kernel(), dg.last_kernel()
    assert parity.worst_ratio(path, got, A, B, C, 1.25, -0.5) <= 1.0


@pytest.mark.parametrize("path", ["tf32", "f16_tn", "bf16_nn"])
def test_pair_wide_integers_bit_exact(path):
    import dense_gemm_09_gb300 as dg
    # several tiles per pair (both accumulator phases), exact integer sums
    A, B, C = parity.host_operands(path, 2048, 3072, 256, seed=9, dist="int")
    dg.tune_next(dg.TUNE_PAIR_WIDE)
    got, _, _ = parity.run(path, A, B, C, 1.0, 1.0)
    assert "_pair_256x512x" in dg.last_kernel()
    ref, _ = parity.reference(path, A, B, C, 1.0, 1.0)
    assert np.array_equal(got.double().numpy(), ref)


# Few output tiles and a long K: the split-K kernel (a cluster of S CTAs per
# tile, partials reduced in distributed shared memory).
SPLITK_CASES = [
    ("f16_tn", (100, 1000, 2048)),   # few tiles: the automatic choice splits K
    ("f16_tn", (64, 512, 1024)),
    ("f16_tn", (300, 512, 4096)),    # M > 128 still splits when tiles are few
    ("f16_tn", (127, 2048, 1000)),   # K tail inside the last range
    ("tf32", (100, 520, 1000)),      # K tail
    ("tf32", (256, 256, 2048)),
    ("f16_nn", (100, 1000, 2048)),
    ("bf16_tn", (127, 2048, 1000)),
    ("bf16_nn", (300, 512, 4096)),
]


@pytest.mark.parametrize("path,shape", SPLITK_CASES)
def test_splitk_kernel(path, shape):
    import dense_gemm_09_gb300 as dg
    M, N, K = shape
    A, B, C = parity.host_operands(path, M, N, K, seed=M * 3 + N)
    got, _, _ = parity.run(path, A, B, C, 1.5, -0.25)
    assert "_splitk" in dg.last_kernel(), dg.last_kernel()
    assert parity.worst_ratio(path, got, A, B, C, 1.5, -0.25) <= 1.0


@pytest.mark.parametrize("path", ["tf32", "f16_tn", "f16_nn"])
def test_splitk_integers_bit_exact(path):
    import dense_gemm_09_gb300 as dg
    M, N, K = 120, 600, 2048
    A, B, C = parity.host_operands(path, M, N, K, seed=31, dist="int")
    got, _, _ = parity.run(path, A, B, C, 1.0, 1.0)
    assert "_splitk" in dg.last_kernel()
    ref, _ = parity.reference(path, A, B, C, 1.0, 1.0)
    assert np.array_equal(got.double().numpy(), ref)


def test_splitk_is_deterministic():
    # the partials are added in rank order, whatever the timing
    import dense_gemm_09_gb300 as dg
    A, B, C = parity.host_operands("f16_tn", 127, 1024, 4096, seed=5)
    outs = [parity.run("f16_tn", A, B, C, 1.0, 0.0)[0] for _ in range(3)]
    assert "_splitk" in dg.last_kernel()
    assert all(torch.equal(outs[0], o) for o in outs[1:])


# FP32 SIMT: a problem with fewer tiles than resident CTAs (2 per SM) runs
# split-K in clusters, the partials added in distributed shared memory.  The
# expected split assumes GB300's 152 SMs (304 resident CTAs).
SIMT_SPLIT_CASES = [
    ((256, 256, 256), "sgemm_simt_splitk8_"),          # 4 tiles, split 8 ways
    ((100, 1000, 2048), "sgemm_simt_splitk8_"),        # 8 tiles, M tail
    ((1000, 1000, 3000), "sgemm_simt_splitk4_"),       # 64 tiles, M/N/K tails
    ((300, 520, 4100), "sgemm_simt_splitk8_"),         # 15 tiles, K tail in the last range
    ((127, 12288, 640), "sgemm_simt_splitk3_"),        # 96 tiles, skinny
    ((1200, 1300, 600), "sgemm_simt_splitk2_"),        # 110 tiles
    ((2048, 2048, 64), "sgemm_simt_tma_"),             # 256 tiles, K too short to split (TMA-fed)
    ((4092, 4092, 512), "sgemm_simt_tma_"),            # more tiles than one wave: no split (TMA-fed)
]


@pytest.mark.parametrize("shape,name", SIMT_SPLIT_CASES)
def test_simt_split_tail(shape, name):
    import dense_gemm_09_gb300 as dg
    M, N, K = shape
    A, B, C = parity.host_operands("f32", M, N, K, seed=M + 3 * N + K)
    got, _, _ = parity.run("f32", A, B, C, 1.5, -0.25)
    assert name in dg.last_kernel(), dg.last_kernel()
    assert parity.worst_ratio("f32", got, A, B, C, 1.5, -0.25) <= 1.0


@pytest.mark.parametrize("shape", [(120, 600, 2048), (1000, 1000, 3000)])
def test_simt_split_integers_bit_exact(shape):
    import dense_gemm_09_gb300 as dg
    M, N, K = shape
    A, B, C = parity.host_operands("f32", M, N, K, seed=37, dist="int")
    got, _, _ = parity.run("f32", A, B, C, 1.0, 2.0)
    assert "splitk" in dg.last_kernel()
    ref, _ = parity.reference("f32", A, B, C, 1.0, 2.0)
    assert np.array_equal(got.double().numpy(), ref)


def test_simt_split_is_deterministic():
    import dense_gemm_09_gb300 as dg
    A, B, C = parity.host_operands("f32", 1000, 1000, 3000, seed=8)
    outs = [parity.run("f32", A, B, C, 1.0, 0.0)[0] for _ in range(3)]
    assert "splitk" in dg.last_kernel()
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_simt_split_unaligned_b():
    # B's pitch is not a multiple of 4 floats: the 4-byte-copy instantiation
    import dense_gemm_09_gb300 as dg
    M, N, K = 300, 257, 3001
    A, B, C = parity.host_operands("f32", M, N, K, seed=41)
    got, _, _ = parity.run("f32", A, B, C, 1.5, -0.25, pad=(0, 2, 0))
    assert dg.last_kernel().startswith("sgemm_simt_splitk") and dg.last_kernel().endswith("cpasync4")
    assert parity.worst_ratio("f32", got, A, B, C, 1.5, -0.25) <= 1.0


# N-major B (TF32 and the NN 16-bit kinds) whose N is not a whole number of
# 128-byte column groups: the pair kernels load every tile column but the
# last with one 3-D box per stage, and the last one with 2-D boxes.
@pytest.mark.parametrize("path", ["tf32", "f16_nn", "bf16_nn"])
# (N a multiple of 8 but not of 64, K a multiple of 8: TMA-describable pitches
# for every kind; K = 312 also leaves a partial last K block)
@pytest.mark.parametrize("shape", [(600, 4088, 256), (520, 1096, 312), (300, 520, 264)])
@pytest.mark.parametrize("wide", [False, True], ids=["256x256", "256x512"])
def test_n_major_ragged_n_pair(path, shape, wide):
    import dense_gemm_09_gb300 as dg
    M, N, K = shape
    A, B, C = parity.host_operands(path, M, N, K, seed=M + 2 * N + K)
    dg.tune_next(dg.TUNE_PAIR_WIDE if wide else dg.TUNE_PAIR, 256, dg.SK_OFF)
    got, _, _ = parity.run(path, A, B, C, 1.25, -0.5)
    assert "_pair_" in dg.last_kernel(), dg.last_kernel()
    assert dg.device_status() == dg.OK
    assert parity.worst_ratio(path, got, A, B, C, 1.25, -0.5) <= 1.0


# FP32 SIMT fed by TMA: problems of at least a wave of tiles whose A and B
# have 16-byte aligned bases and pitches.  Tails in M, N and K come from TMA's
# zero fill and the epilogue's masks; a C pitch that is not a multiple of 4
# takes the scalar stores.
SIMT_TMA_CASES = [
    ((2049, 2561, 1001), (3, 3, 0)),   # M, N, K tails; lda 1004, ldb 2564; C pitch 2561
    ((2100, 2500, 37), (3, 0, 0)),     # K = 37: one partial K slice
    ((2176, 2304, 96), (0, 0, 4)),     # whole tiles; padded C
    ((4092, 4092, 512), (0, 0, 0)),    # the 4092 workload's shape with a shorter K
]


@pytest.mark.parametrize("shape,pad", SIMT_TMA_CASES)
def test_simt_tma_kernel_matches_oracle(shape, pad):
    import dense_gemm_09_gb300 as dg
    M, N, K = shape
    A, B, C = parity.host_operands("f32", M, N, K, seed=M + N + 7 * K)
    got, _, _ = parity.run("f32", A, B, C, 1.5, -0.25, pad=pad)
    assert dg.last_kernel().startswith("sgemm_simt_tma_"), dg.last_kernel()
    assert parity.worst_ratio("f32", got, A, B, C, 1.5, -0.25) <= 1.0


def test_simt_tma_kernel_is_bit_identical_to_cp_async_kernel():
    # the same FMAs in the same order: A with an odd pitch takes the cp.async
    # kernel, the aligned copy the TMA-fed one
    import dense_gemm_09_gb300 as dg
    M, N, K = 2100, 2400, 700
    A, B, C = parity.host_operands("f32", M, N, K, seed=77)
    tma, _, _ = parity.run("f32", A, B, C, 0.75, 0.5)
    assert dg.last_kernel().startswith("sgemm_simt_tma_"), dg.last_kernel()
    cpa, _, _ = parity.run("f32", A, B, C, 0.75, 0.5, pad=(1, 0, 0))
    assert dg.last_kernel().startswith("sgemm_simt_128x128"), dg.last_kernel()
    assert torch.equal(tma, cpa)


def test_simt_tma_integers_bit_exact():
    import dense_gemm_09_gb300 as dg
    A, B, C = parity.host_operands("f32", 2304, 2176, 1028, seed=38, dist="int")
    got, _, _ = parity.run("f32", A, B, C, 1.0, 2.0)
    assert dg.last_kernel().startswith("sgemm_simt_tma_"), dg.last_kernel()
    ref, _ = parity.reference("f32", A, B, C, 1.0, 2.0)
    assert np.array_equal(got.double().numpy(), ref)


# The tuning hook: every tile configuration the sweep tool can request gives
# a correct result (narrow tiles, tiles whose width is not a multiple of the
# TMA-store box, every split factor, and splits wider than K allows).
def _tune_cases():
    import dense_gemm_09_gb300 as dg
    cases = []
    for path in ("f16_tn", "tf32"):
        cases += [(path, (300, 1000, 1024), dg.TUNE_PAIR, 256, 1)]
        cases += [(path, (200, 1000, 1024), dg.TUNE_SINGLE, bn, 1) for bn in (32, 96, 160, 224, 256)]
        cases += [(path, (127, 1000, 2048), dg.TUNE_SPLIT, bn, S) for bn, S in
                  ((32, 2), (96, 3), (128, 4), (160, 5), (192, 6), (224, 7), (256, 8))]
        cases += [(path, (100, 300, 200), dg.TUNE_SPLIT, 64, 8)]  # 4 or 7 K blocks: S lowered
    # N = 520 keeps the NN kinds' B pitch a multiple of 16 bytes (TMA, so the pair can run)
    cases += [(path, (255, 520, 304), dg.TUNE_PAIR, 256, 1) for path in parity.TC_PATHS]
    cases += [("f16_nn", (200, 1000, 1024), dg.TUNE_SINGLE, 192, 1),
              ("f16_nn", (127, 1000, 2048), dg.TUNE_SPLIT, 128, 3),
              ("bf16_nn", (127, 1000, 2048), dg.TUNE_SPLIT, 64, 2),
              ("bf16_tn", (200, 1000, 1024), dg.TUNE_SINGLE, 96, 1)]
    return cases


@pytest.mark.parametrize("path,shape,variant,bn,split", _tune_cases())
def test_tuned_configurations(path, shape, variant, bn, split):
    import dense_gemm_09_gb300 as dg
    M, N, K = shape
    A, B, C = parity.host_operands(path, M, N, K, seed=M + N + bn + split)
    dg.tune_next(variant, bn, split)
    got, _, _ = parity.run(path, A, B, C, 1.5, -0.25)
    name = dg.last_kernel()
    if variant == dg.TUNE_PAIR:
        assert "_pair_" in name
    else:
        assert ("_128x%dx" % bn) in name, name
        assert ("_splitk" in name) == (variant == dg.TUNE_SPLIT), name
    assert parity.worst_ratio(path, got, A, B, C, 1.5, -0.25) <= 1.0


def test_tuning_is_one_shot():
    import dense_gemm_09_gb300 as dg
    A, B, C = parity.host_operands("f16_tn", 127, 1000, 2048, seed=6)
    dg.tune_next(dg.TUNE_PAIR)
    parity.run("f16_tn", A, B, C, 1.0, 0.0)
    assert "_pair_" in dg.last_kernel()
    parity.run("f16_tn", A, B, C, 1.0, 0.0)  # M = 127: the automatic choice is never the pair
    assert "_pair_" not in dg.last_kernel()
