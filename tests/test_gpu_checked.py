"""The checked build (libdgemm_checked.so, compiled with -DDGEMM_CHECKED).

Every kernel of that build tests the indices it computes -- shared-memory
offsets, tile coordinates, global rows and columns, 16-byte alignment, TMEM
columns, workspace regions -- and a failed check skips its access and records
DGEMM_ERR_BOUNDS with its site instead of trapping.  This stands in for a
memory checker on a pool where none can run.

The odd shapes of the parity tests (1..9, 15..17, 31..33, 127..129 and a few
multi-tile ones) go through the checked library's C ABI on every path and
every kernel family (SIMT cp.async and TMA-fed, split-K, the CTA pair with
and without the stream-K tail, the single-CTA kernel, the register-path and
cp.async producers, the workspace copies): each result must agree with the
oracle and no check may fail.  A negative control shows that the checks are
live: a test hook narrows one bound, and the stores past it are skipped and
reported, with nothing written there.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Lc():
    import dense_gemm_09_gb300 as dg
    from dense_gemm_09_gb300 import _build
    _build.build(checked=True)  # no-op when build() made it already
    L = dg.lib_checked()
    torch.cuda.synchronize()
    assert L.dgemm_device_status(1) == dg.OK
    return L


def _call(L, path, dA, dB, dC, alpha, beta):
    M, K = dA.shape
    N = dC.shape[1]
    fn = getattr(L, parity.fn(path).__name__)
    return fn(M, N, K, ctypes.c_float(alpha), dA.data_ptr(), dA.stride(0), dB.data_ptr(), dB.stride(0),
              ctypes.c_float(beta), dC.data_ptr(), dC.stride(0),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _check(L, path, shape, pad=(0, 0, 0), tune=None, alpha=1.5, beta=-0.25, seed=0):
    import dense_gemm_09_gb300 as dg
    M, N, K = shape
    A, B, C = parity.host_operands(path, M, N, K, seed=seed or (M * 3 + N * 5 + K))
    dA, _ = parity.to_device_padded(A, pad[0])
    dB, _ = parity.to_device_padded(B, pad[1])
    dC, _ = parity.to_device_padded(C, pad[2], fill=float("nan") if pad[2] else 0.0)
    if tune is not None:
        assert L.dgemm_tune_next(*tune) == dg.OK
    assert _call(L, path, dA, dB, dC, alpha, beta) == dg.OK
    st = L.dgemm_device_status(0)
    site = L.dgemm_check_site()
    L.dgemm_device_status(1)
    name = L.dgemm_last_kernel().decode()
    assert st == dg.OK and site == 0, "%s: %s at site %d" % (name, dg.status_string(st), site)
    assert parity.worst_ratio(path, dC.cpu(), A, B, C, alpha, beta) <= 1.0, name
    return name


ODD = [1, 2, 3, 5, 7, 9, 15, 16, 17, 31, 32, 33, 127, 128, 129]


def _odd_shapes(n=24, seed=5):
    rng = np.random.default_rng(seed)
    return [tuple(int(rng.choice(ODD)) for _ in range(3)) for _ in range(n)]


@pytest.mark.parametrize("path", parity.PATHS)
@pytest.mark.parametrize("pad", [(0, 0, 0), (1, 3, 2)], ids=["tight", "padded"])
def test_odd_shapes_pass_every_check(Lc, path, pad):
    for shape in _odd_shapes():
        _check(Lc, path, shape, pad=pad)


# Larger problems, one per kernel family: (path, shape, pad, tuning, name fragment)
FAMILIES = [
    ("f32", (2049, 2561, 1001), (3, 3, 0), None, "sgemm_simt_tma_"),      # TMA-fed SIMT, tails
    ("f32", (1000, 1000, 3000), (0, 0, 0), None, "sgemm_simt_splitk"),    # SIMT split-K clusters
    ("f32", (2100, 2500, 301), (1, 0, 0), None, "sgemm_simt_128x128"),    # SIMT cp.async kernel
    ("f16_tn", (600, 1100, 520), (0, 0, 0), (1, 256, 1), "_pair_256x256"),   # CTA pair, whole tiles
    ("tf32", (2500, 4500, 1000), (0, 0, 0), (5, 256, 2), "_sk_"),         # wide pair, stream-K tail
    ("f16_tn", (2304, 2304, 512), (0, 0, 0), (1, 256, 2), "_sk_"),        # pair, stream-K tail
    ("bf16_nn", (300, 704, 200), (0, 0, 0), (2, 128, 1), "_128x128"),     # single-CTA kernel
    ("f16_tn", (100, 1000, 2048), (0, 0, 0), None, "_splitk"),            # split-K in clusters (DSMEM)
    ("f16_tn", (100, 1000, 520), (0, 0, 0), (8, 192, 1), "_pair_128x192"),  # small-M pair, ragged N
    ("tf32", (40, 2048, 264), (0, 0, 0), (8, 256, 1), "_pair_128x256"),     # small-M pair, N-major B
    ("tf32", (300, 520, 130), (1, 2, 0), None, "_cpasync"),               # cp.async producer
    ("f16_nn", (300, 520, 130), (1, 2, 0), None, "_ldst"),                # register-path producer
    ("f16_tn", (257, 300, 72), (0, 0, 3), None, "umma_f16_tn"),           # unaligned C: row-by-row stores
]


@pytest.mark.parametrize("path,shape,pad,tune,frag", FAMILIES, ids=[f[4].strip("_") + "-" + f[0] for f in FAMILIES])
def test_kernel_families_pass_every_check(Lc, path, shape, pad, tune, frag):
    name = _check(Lc, path, shape, pad=pad, tune=tune)
    assert frag in name, name


def test_fuzz_cases_pass_every_check(Lc):
    """Every fourth seeded case of the general fuzz (all paths, pitch padding,
    base offsets, forced tile configurations) through the checked library."""
    import dense_gemm_09_gb300 as dg
    from tests.test_gpu_fuzz import CASES
    for path, (M, N, K), pad, offset, alpha, beta, tune in CASES[::4]:
        A, B, C = parity.host_operands(path, M, N, K, seed=M * 7 + N * 13 + K)
        dA, _ = parity.to_device_padded(A, pad[0], offset_elems=offset[0])
        dB, _ = parity.to_device_padded(B, pad[1], offset_elems=offset[1])
        dC, _ = parity.to_device_padded(C, pad[2], fill=float("nan") if pad[2] else 0.0, offset_elems=offset[2])
        if tune[0] != 0:
            assert Lc.dgemm_tune_next(*tune) == dg.OK
        assert _call(Lc, path, dA, dB, dC, alpha, beta) == dg.OK
        st, site = Lc.dgemm_device_status(0), Lc.dgemm_check_site()
        Lc.dgemm_device_status(1)
        name = Lc.dgemm_last_kernel().decode()
        assert st == dg.OK and site == 0, "%s %s: %s at site %d" % (path, (M, N, K), name, site)
        assert parity.worst_ratio(path, dC.cpu(), A, B, C, alpha, beta) <= 1.0, name


def test_workspace_copies_pass_every_check(Lc):
    import dense_gemm_09_gb300 as dg
    M, N, K = 301, 257, 129
    A, B, C = parity.host_operands("tf32", M, N, K, seed=12)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    need = Lc.gemm_tf32_workspace_bytes(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = Lc.gemm_tf32_ws(M, N, K, ctypes.c_float(1.0), dA.data_ptr(), K, dB.data_ptr(), N, ctypes.c_float(0.5),
                         dC.data_ptr(), N, ws.data_ptr(), need, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == dg.OK
    assert Lc.dgemm_device_status(0) == dg.OK and Lc.dgemm_check_site() == 0
    assert parity.worst_ratio("tf32", dC.cpu(), A, B, C, 1.0, 0.5) <= 1.0


def test_a_narrowed_bound_is_caught_and_its_stores_skipped(Lc):
    """Negative control: the hook makes the next TMA-fed SIMT launch check its
    C stores against M - 3 rows; those stores fail, are skipped (C keeps its
    old values there) and are reported with a site in sgemm_tma.cu."""
    import dense_gemm_09_gb300 as dg
    M, N, K = 2048, 2560, 64
    A, B, C = parity.host_operands("f32", M, N, K, seed=13)
    dA, dB = A.cuda(), B.cuda()
    dC = torch.full((M, N), 7.0, device="cuda")
    assert Lc.dgemm_test_shrink_bounds(3) == dg.OK
    assert _call(Lc, "f32", dA, dB, dC, 1.0, 0.0) == dg.OK
    assert Lc.dgemm_last_kernel().decode().startswith("sgemm_simt_tma_")
    st = Lc.dgemm_device_status(0)
    site = Lc.dgemm_check_site()
    assert Lc.dgemm_device_status(1) == dg.ERR_BOUNDS
    assert st == dg.ERR_BOUNDS
    assert site // 100000 == 2, site  # unit 2: sgemm_tma.cu
    out = dC.cpu()
    assert bool((out[M - 3:] == 7.0).all())  # skipped
    Cz = torch.zeros_like(C)
    assert parity.worst_ratio("f32", out[:M - 3], A[:M - 3], B, Cz[:M - 3], 1.0, 0.0) <= 1.0
    # the next launch has the full bound again
    assert _call(Lc, "f32", dA, dB, dC, 1.0, 0.0) == dg.OK
    assert Lc.dgemm_device_status(1) == dg.OK and Lc.dgemm_check_site() == 0


def test_normal_build_reports_no_site():
    # libdgemm.so compiles the checks out: the site is always 0 and the hook
    # changes nothing
    import dense_gemm_09_gb300 as dg
    L = dg.lib()
    M, N, K = 2048, 2560, 64
    A, B, C = parity.host_operands("f32", M, N, K, seed=14)
    dA, dB, dC = A.cuda(), B.cuda(), torch.zeros((M, N), device="cuda")
    assert L.dgemm_test_shrink_bounds(5) == dg.OK
    dg.gemm_f32(dA, dB, dC, 1.0, 0.0)
    assert dg.device_status() == dg.OK and L.dgemm_check_site() == 0
    assert parity.worst_ratio("f32", dC.cpu(), A, B, torch.zeros_like(C), 1.0, 0.0) <= 1.0
