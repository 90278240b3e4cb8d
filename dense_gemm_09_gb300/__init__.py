"""Python binding of libdgemm (include/dgemm.h): dense row-major GEMM on GB300.

Argument marshalling only: every entry point takes torch CUDA tensors, reads
their data pointers, row pitches and the current stream, and calls the C ABI
of the same name.  All arithmetic runs in the library's CUDA kernels; there
is no fallback of any kind -- if the library is missing or the call fails,
an exception is raised.

    gemm_f32(A, B, C, alpha, beta)     C = alpha*A@B + beta*C     (FP32, CUDA cores)
    gemm_tf32(A, B, C, alpha, beta)    same, TF32 tensor cores   (FP32 in / out)
    gemm_f16_tn(A, B, C, alpha, beta)  C = alpha*A@B.T + beta*C  (FP16 in / out,
                                                                   FP32 accumulate)
    gemm_f16_nn(A, B, C, alpha, beta)  C = alpha*A@B + beta*C    (FP16, B is K x N)
    gemm_bf16_tn / gemm_bf16_nn         the same with bfloat16

Matrices are 2-D tensors with unit column stride; a row stride larger than
the width is passed on as the leading dimension.  C is updated in place and
returned.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdgemm.so")
LIB_CHECKED_PATH = os.path.join(_PKG, "libdgemm_checked.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_DEVICE, ERR_LAUNCH, ERR_TIMEOUT, ERR_BOUNDS = 0, 1, 2, 3, 4, 5

_lock = threading.Lock()
_lib = None
_lib_checked = None


class DgemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, status_string(status)))


def build(force: bool = False) -> str:
    """Compile libdgemm.so and the checked build libdgemm_checked.so (nvcc,
    sm_103a) in-tree; returns the path of libdgemm.so."""
    from . import _build
    return _build.build_all(force=force)[0]


def lib():
    """The loaded C library, with its signatures declared."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(LIB_PATH)
        return _lib


def lib_checked():
    """The checked build (same ABI; device-side bounds checks compiled in),
    loaded beside the normal library, with its signatures declared."""
    global _lib_checked
    with _lock:
        if _lib_checked is None:
            _lib_checked = _load(LIB_CHECKED_PATH)
        return _lib_checked


def _load(path: str):
    if not os.path.exists(path):
        raise RuntimeError("%s is not built; run dense_gemm_09_gb300.build()" % path)
    L = ctypes.CDLL(path)
    i64, f32, vp, ci = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
    sig = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
    for name in ("gemm_f32", "gemm_tf32", "gemm_f16_tn", "gemm_f16_nn", "gemm_bf16_tn",
                 "gemm_bf16_nn"):
        fn = getattr(L, name)
        fn.argtypes = sig
        fn.restype = ci
    L.dgemm_status_string.argtypes = [ci]
    L.dgemm_status_string.restype = ctypes.c_char_p
    L.dgemm_device_status.argtypes = [ci]
    L.dgemm_device_status.restype = ci
    L.dgemm_test_inject_stall.argtypes = [ctypes.c_uint64]
    L.dgemm_test_inject_stall.restype = ci
    L.dgemm_last_kernel.argtypes = []
    L.dgemm_last_kernel.restype = ctypes.c_char_p
    L.dgemm_tune_next.argtypes = [ci, ci, ci]
    L.dgemm_tune_next.restype = ci
    L.gemm_tf32_ws.argtypes = sig[:11] + [vp, i64, vp]
    L.gemm_tf32_ws.restype = ci
    L.gemm_f32_ws.argtypes = sig[:11] + [vp, i64, vp]
    L.gemm_f32_ws.restype = ci
    L.gemm_tf32_workspace_bytes.argtypes = [i64, i64, i64, vp, i64, vp, i64]
    L.gemm_tf32_workspace_bytes.restype = i64
    L.gemm_tf32_noalloc.argtypes = sig
    L.gemm_tf32_noalloc.restype = ci
    L.dgemm_test_pair_units.argtypes = [i64, i64, i64, i64, i64, vp, i64]
    L.dgemm_test_pair_units.restype = i64
    L.dgemm_test_stream_k_tiles.argtypes = [i64, i64, i64, ci, ci]
    L.dgemm_test_stream_k_tiles.restype = i64
    L.dgemm_test_choose_config.argtypes = [ci, i64, i64, i64, ci, vp, vp, vp]
    L.dgemm_test_choose_config.restype = ci
    L.dgemm_check_site.argtypes = []
    L.dgemm_check_site.restype = ci
    L.dgemm_test_shrink_bounds.argtypes = [i64]
    L.dgemm_test_shrink_bounds.restype = ci
    return L


def status_string(status: int) -> str:
    return lib().dgemm_status_string(int(status)).decode()


def device_status(clear: bool = True) -> int:
    """The kernels' device status word (synchronises the device)."""
    return lib().dgemm_device_status(1 if clear else 0)


def test_inject_stall(wait_limit_ns: int) -> None:
    """Test hook: the next tensor-core launch on this thread stalls on purpose
    and its bounded waits (limit wait_limit_ns) run out; see include/dgemm.h."""
    lib().dgemm_test_inject_stall(int(wait_limit_ns))


# Tile configurations for tune_next (see dgemm_tune_next in include/dgemm.h)
TUNE_AUTO, TUNE_PAIR, TUNE_SINGLE, TUNE_SPLIT, TUNE_PAIR_WIDE = 0, 1, 2, 3, 5
# the CTA-pair variants with the finer stage ring (K-major 16-bit calls)
TUNE_PAIR_FINE, TUNE_PAIR_WIDE_FINE = 6, 7
# the CTA pair for small M: 128 x bn tiles (bn 128, 192 or 256), 64 rows of A per CTA
TUNE_PAIR128 = 8
# `split` of the CTA-pair variants (TUNE_PAIR, TUNE_PAIR_WIDE): stream-K tail
# chosen automatically, never, or whenever the tiles outnumber the pairs
SK_AUTO, SK_OFF, SK_ON = 0, 1, 2


def tune_next(variant: int, bn: int = 256, split: int = 1) -> None:
    """Tuning hook: fix the tile configuration of the next tensor-core call
    on this thread (variant TUNE_PAIR / TUNE_PAIR_WIDE / TUNE_PAIR_FINE /
    TUNE_PAIR_WIDE_FINE / TUNE_SINGLE / TUNE_SPLIT / TUNE_PAIR128, tile width bn, split-K
    factor split; for the pair variants, split is the stream-K mode SK_*)."""
    st = lib().dgemm_tune_next(int(variant), int(bn), int(split))
    if st != OK:
        raise DgemmError(st, "dgemm_tune_next")


def last_kernel() -> str:
    """Name of the kernel variant the last call on this thread launched."""
    return lib().dgemm_last_kernel().decode()


def _mat(t: torch.Tensor, name: str, dtype: torch.dtype):
    if not isinstance(t, torch.Tensor) or t.dim() != 2:
        raise ValueError("%s must be a 2-D tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    rows, cols = t.shape
    if cols > 1 and t.stride(1) != 1:
        raise ValueError("%s must have unit column stride" % name)
    # the row stride as stored, also for one row (it decides whether the TMA
    # kernels can load the matrix); never below the row length
    ld = t.stride(0) if rows > 0 else cols
    return t.data_ptr(), max(ld, cols)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _call(name, M, N, K, alpha, pa, lda, pb, ldb, beta, pc, ldc, stream):
    st = getattr(lib(), name)(M, N, K, float(alpha), pa, lda, pb, ldb, float(beta), pc, ldc,
                              _stream(stream))
    if st != OK:
        raise DgemmError(st, name)


def _nn(name, A, B, C, alpha, beta, stream):
    pa, lda = _mat(A, "A", torch.float32)
    pb, ldb = _mat(B, "B", torch.float32)
    pc, ldc = _mat(C, "C", torch.float32)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError("shape mismatch: A %s, B %s, C %s" % (tuple(A.shape), tuple(B.shape), tuple(C.shape)))
    _call(name, M, N, K, alpha, pa, lda, pb, ldb, beta, pc, ldc, stream)
    return C


def gemm_f32(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C = alpha * A @ B + beta * C on the FP32 pipes (A: M x K, B: K x N)."""
    return _nn("gemm_f32", A, B, C, alpha, beta, stream)


def gemm_tf32(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C = alpha * A @ B + beta * C with TF32 tensor-core products."""
    return _nn("gemm_tf32", A, B, C, alpha, beta, stream)


def tf32_workspace_bytes(A, B) -> int:
    """Bytes of workspace gemm_tf32_ws needs for these operands (0: none)."""
    pa, lda = _mat(A, "A", torch.float32)
    pb, ldb = _mat(B, "B", torch.float32)
    M, K = A.shape
    n = lib().gemm_tf32_workspace_bytes(M, B.shape[1], K, pa, lda, pb, ldb)
    if n < 0:
        raise DgemmError(ERR_INVALID_ARG, "gemm_tf32_workspace_bytes")
    return int(n)


def _ws_call(name, A, B, C, alpha, beta, workspace, stream):
    pa, lda = _mat(A, "A", torch.float32)
    pb, ldb = _mat(B, "B", torch.float32)
    pc, ldc = _mat(C, "C", torch.float32)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError("shape mismatch: A %s, B %s, C %s" % (tuple(A.shape), tuple(B.shape), tuple(C.shape)))
    pw, nw = 0, 0
    if workspace is not None:
        if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda:
            raise ValueError("workspace must be a CUDA tensor")
        pw, nw = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = getattr(lib(), name)(M, N, K, float(alpha), pa, lda, pb, ldb, float(beta), pc, ldc,
                              pw or None, nw, _stream(stream))
    if st != OK:
        raise DgemmError(st, name)
    return C


def gemm_tf32_ws(A, B, C, alpha: float = 1.0, beta: float = 0.0, workspace=None, stream=None):
    """gemm_tf32 for operands whose base or row pitch TMA cannot load: they
    are copied into ``workspace`` (a CUDA tensor of at least
    tf32_workspace_bytes(A, B) bytes, 16-byte aligned) first."""
    return _ws_call("gemm_tf32_ws", A, B, C, alpha, beta, workspace, stream)


def gemm_f32_ws(A, B, C, alpha: float = 1.0, beta: float = 0.0, workspace=None, stream=None):
    """gemm_f32 with the same workspace: a B whose base or row pitch is not a
    16-byte multiple is copied first, so the SIMT kernel loads it in 16-byte
    pieces."""
    return _ws_call("gemm_f32_ws", A, B, C, alpha, beta, workspace, stream)


# Bytes of the library's fixed scratch behind gemm_tf32_noalloc (see
# DGEMM_NOALLOC_SCRATCH_BYTES in include/dgemm.h).
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def gemm_tf32_noalloc(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """gemm_tf32_ws for callers that cannot allocate device memory: the
    copies of operands TMA cannot load go to a fixed 64 MiB scratch array
    inside the library instead of a caller workspace.  Calls that overlap on
    the GPU share that array and race; operands whose copies need more than
    NOALLOC_SCRATCH_BYTES are refused."""
    need = tf32_workspace_bytes(A, B)
    if need > NOALLOC_SCRATCH_BYTES:
        raise DgemmError(ERR_INVALID_ARG, "gemm_tf32_noalloc (the operands' padded copies need %d bytes; "
                         "the fixed scratch holds %d)" % (need, NOALLOC_SCRATCH_BYTES))
    return _nn("gemm_tf32_noalloc", A, B, C, alpha, beta, stream)


def _gemm16(name, dtype, tn, A, B, C, alpha, beta, stream):
    pa, lda = _mat(A, "A", dtype)
    pb, ldb = _mat(B, "B", dtype)
    pc, ldc = _mat(C, "C", dtype)
    M, K = A.shape
    N, K2 = B.shape if tn else (B.shape[1], B.shape[0])
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError("shape mismatch: A %s, B %s, C %s" % (tuple(A.shape), tuple(B.shape), tuple(C.shape)))
    _call(name, M, N, K, alpha, pa, lda, pb, ldb, beta, pc, ldc, stream)
    return C


def gemm_f16_tn(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C = alpha * A @ B.T + beta * C; A: M x K, B: N x K, C: M x N, all f16."""
    return _gemm16("gemm_f16_tn", torch.float16, True, A, B, C, alpha, beta, stream)


def gemm_f16_nn(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C = alpha * A @ B + beta * C; A: M x K, B: K x N, C: M x N, all f16."""
    return _gemm16("gemm_f16_nn", torch.float16, False, A, B, C, alpha, beta, stream)


def gemm_bf16_tn(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C = alpha * A @ B.T + beta * C with bfloat16 A, B (N x K) and C."""
    return _gemm16("gemm_bf16_tn", torch.bfloat16, True, A, B, C, alpha, beta, stream)


def gemm_bf16_nn(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C = alpha * A @ B + beta * C with bfloat16 A, B (K x N) and C."""
    return _gemm16("gemm_bf16_nn", torch.bfloat16, False, A, B, C, alpha, beta, stream)
