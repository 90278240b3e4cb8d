"""CPU oracle for dense row-major GEMM ``C = alpha*A*B + beta*C``.

TEST INFRASTRUCTURE ONLY.  The product (the CUDA library and its Python
binding) never imports, loads or calls anything in this package.  Only the
test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
use it.  It shares no code with the CUDA path; the arithmetic lives in
``dgemm_oracle.c`` (plain C, double accumulation, a triple loop).

Sources (page title, section):
  * "SGEMM CUDA代码学习", "问题定义与记号" -- row-major C = A x B, one output
    element is one K-long dot product.
  * "CUDA GEMM：从基础写法到工程优化", opening definition -- C = alpha*A*B + beta*C.
  * "SGEMM CUDA代码学习", "第 5 步" -- TF32 is 1+8+10 bits.
  * "Warp Specialization HGEMM", "6. B 的 RowMajor(K,N) 与 TN 布局" -- the TN
    layout: B is stored N x K and C = A * B^T.
  * "HGEMM SMEM Swizzle 代码学习", the kernel source's layout notes -- NN: A, B,
    C all row-major; TN: B stored N x K.
  * "SGEMM CUDA代码学习", "第 5 步" -- BF16 among the tensor-core precisions.

Acceptance, per element (the tolerance rule results are checked against):
    |C_gpu - ref| <= tol * (|A||B|)_ij + tol * |beta * c_ij|
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dgemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, TF32_NEAREST_AWAY, TF32_TRUNCATE, F16, BF16 = 0, 1, 2, 3, 4
_KIND = {"f32": F32, "tf32": TF32_NEAREST_AWAY, "tf32_rna": TF32_NEAREST_AWAY,
         "tf32_rz": TF32_TRUNCATE, "f16": F16, "bf16": BF16}

# Acceptance tolerances per path (relative to |A||B| and |beta*C|).
def tol_f32(K: int) -> float:
    return 1e-6 * max(K, 1) ** 0.5


TOL_TF32 = 2e-3
TOL_F16 = 1e-3
# BF16 (no tolerance is fixed for it): bfloat16 keeps 8 significant bits, so
# the single rounding of the result costs up to half an ulp, 2^-8 of |result|
# <= 2^-8 * (|alpha| |A||B| + |beta c|) -- at most 1.5 * 2^-8 = 5.9e-3 of the
# bound's terms for |alpha| <= 1.5; FP32 accumulation adds ~K * 2^-24.
TOL_BF16 = 8e-3

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math) into liboracle.so."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                           "-pthread", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def load_library(path: str):
    """Open a compiled oracle and declare its C signatures."""
    lib = ctypes.CDLL(path)
    i64, dbl, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    lib.oracle_f16_value.restype = dbl
    lib.oracle_f16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_value.restype = dbl
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_tf32_value.restype = dbl
    lib.oracle_tf32_value.argtypes = [ctypes.c_float, ctypes.c_int]
    lib.oracle_widen.restype = None
    lib.oracle_widen.argtypes = [ctypes.c_int, vp, i64, i64, i64, ctypes.c_int, vp]
    lib.oracle_gemm.restype = ctypes.c_int
    lib.oracle_gemm.argtypes = [i64, i64, i64, dbl, vp, vp, dbl, vp,
                                ctypes.c_int, i64, vp, vp, vp, vp, ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
        return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def f16_value(bits: int) -> float:
    """The value of one IEEE binary16 bit pattern."""
    return _load().oracle_f16_value(bits)


def bf16_value(bits: int) -> float:
    """The value of one bfloat16 bit pattern."""
    return _load().oracle_bf16_value(bits)


def tf32_value(x: float, mode: str = "tf32_rna") -> float:
    """One float reduced to TF32 (mode 'tf32_rna' or 'tf32_rz')."""
    return _load().oracle_tf32_value(x, _KIND[mode])


def widen(kind: str, m: np.ndarray, trans: bool = False) -> np.ndarray:
    """Dense float64 copy of the logical operand.

    ``m`` is a 2-D array (float32 for f32/tf32 kinds, float16 or uint16 for
    f16) whose rows may be padded (a row stride above its width).  With
    ``trans`` the logical matrix is m^T (the TN store of B)."""
    code = _KIND[kind]
    if code in (F16, BF16):
        if m.dtype == np.float16:
            m = m.view(np.uint16)
        assert m.dtype == np.uint16
    else:
        assert m.dtype == np.float32
    assert m.ndim == 2
    if m.size and m.shape[1] > 1:
        assert m.strides[1] == m.itemsize
    ld = m.strides[0] // m.itemsize if m.shape[0] > 1 and m.size else m.shape[1]
    rows, cols = (m.shape[1], m.shape[0]) if trans else m.shape
    out = np.empty((rows, cols), dtype=np.float64)
    if out.size:
        _load().oracle_widen(code, _ptr(m), rows, cols, ld, int(trans), _ptr(out))
    return out


def gemm(A64: np.ndarray, B64: np.ndarray, C64, alpha: float, beta: float, *,
         rows=None, cols=None, entries=None, nthreads: int = 0):
    """Reference outputs from widened operands (see :func:`widen`).

    Exactly one of ``rows`` (row indices -> (len, N) arrays), ``cols``
    (column indices -> (len, M) arrays, column u in row u) or ``entries``
    ((i, j) index arrays -> flat arrays) may be given; with none, the full
    M x N product is returned.  Returns ``(ref, absprod)``: the reference
    value alpha*sum(a*b) + beta*c and sum(|a|*|b|), both float64."""
    M, K = A64.shape
    K2, N = B64.shape
    assert K == K2
    A64 = np.ascontiguousarray(A64, dtype=np.float64)
    B64 = np.ascontiguousarray(B64, dtype=np.float64)
    cptr = None
    if beta != 0.0:
        C64 = np.ascontiguousarray(C64, dtype=np.float64)
        assert C64.shape == (M, N)
        cptr = _ptr(C64)
    if entries is not None:
        ii = np.ascontiguousarray(entries[0], dtype=np.int64)
        jj = np.ascontiguousarray(entries[1], dtype=np.int64)
        assert ii.shape == jj.shape
        mode, count, shape = 2, ii.size, (ii.size,)
        assert count == 0 or (ii.min() >= 0 and ii.max() < M and jj.min() >= 0 and jj.max() < N)
    elif cols is not None:
        jj = np.ascontiguousarray(cols, dtype=np.int64)
        ii = jj
        mode, count, shape = 1, jj.size, (jj.size, M)
        assert count == 0 or (jj.min() >= 0 and jj.max() < N)
    else:
        ii = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        jj = ii
        mode, count, shape = 0, ii.size, (ii.size, N)
        assert count == 0 or (ii.min() >= 0 and ii.max() < M)
    ref = np.zeros(shape, dtype=np.float64)
    absprod = np.zeros(shape, dtype=np.float64)
    if count:
        _load().oracle_gemm(M, N, K, float(alpha), _ptr(A64), _ptr(B64), float(beta),
                            cptr, mode, count, _ptr(ii), _ptr(jj), _ptr(ref),
                            _ptr(absprod), int(nthreads))
    return ref, absprod


def reference(kind: str, A: np.ndarray, B: np.ndarray, C, alpha: float, beta: float,
              *, tn: bool = False, **select):
    """Widen the stored operands for path ``kind`` and evaluate the product.

    kind: 'f32', 'tf32_rna', 'tf32_rz', 'f16' or 'bf16' (16-bit operands as
    uint16 bit patterns or float16).  ``tn`` is the layout flag (B stored
    N x K).  C is widened as stored (f32, or the 16-bit kind) and ignored when
    beta == 0."""
    ck = kind if kind in ("f16", "bf16") else "f32"
    A64 = widen(kind, A)
    B64 = widen(kind, B, trans=tn)
    C64 = widen(ck, C) if beta != 0.0 else None
    return gemm(A64, B64, C64, alpha, beta, **select)


def violation_ratio(got, ref, absprod, beta: float, c_old, tol: float) -> np.ndarray:
    """|got - ref| / (tol*|A||B| + tol*|beta*c|), elementwise (<= 1 passes).

    An exact match gives 0 even where the bound is 0; a mismatch against a
    zero bound gives inf."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bound = tol * absprod
    if beta != 0.0:
        bound = bound + tol * np.abs(beta * np.asarray(c_old, dtype=np.float64))
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(err == 0.0, 0.0, err / bound)
    r = np.where(np.isnan(got) != np.isnan(ref), np.inf, r)
    return r
