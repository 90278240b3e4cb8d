"""Helpers for the GPU parity tests: run a path through the C ABI binding on
seeded host operands and compare with the CPU oracle element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import seeded_inputs as si

PATHS = ("f32", "tf32", "f16_tn", "f16_nn", "bf16_tn", "bf16_nn")
TC_PATHS = PATHS[1:]          # tensor-core paths
PATHS16 = PATHS[2:]           # 16-bit operand paths


def is_tn(path: str) -> bool:
    return path.endswith("_tn")


def dtype(path: str) -> torch.dtype:
    return {"f16": torch.float16, "bf1": torch.bfloat16}.get(path[:3], torch.float32)


def fn(path: str):
    import dense_gemm_09_gb300 as dg
    return {"f32": dg.gemm_f32, "tf32": dg.gemm_tf32, "f16_tn": dg.gemm_f16_tn,
            "f16_nn": dg.gemm_f16_nn, "bf16_tn": dg.gemm_bf16_tn, "bf16_nn": dg.gemm_bf16_nn}[path]


def tolerance(path: str, K: int) -> float:
    return {"f32": oracle.tol_f32(K), "tf32": oracle.TOL_TF32}.get(
        path, oracle.TOL_BF16 if path.startswith("bf16") else oracle.TOL_F16)


def oracle_kind(path: str) -> str:
    # TF32: the kernel feeds the stored FP32 operands to the tensor core,
    # which keeps their top 19 bits (truncation toward zero, measured with
    # crafted operands -- see test_tf32_operand_rounding_is_truncation); the
    # oracle reduces operands the same way.
    if path.startswith("bf16"):
        return "bf16"
    if path.startswith("f16"):
        return "f16"
    return {"f32": "f32", "tf32": "tf32_rz"}[path]


def np_operand(t: torch.Tensor) -> np.ndarray:
    """Host tensor -> the array the oracle widens (bfloat16 as raw bits)."""
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def host_operands(path, M, N, K, seed=0, dist="uniform", c_zero=False):
    """Seeded host A (M x K), B (N x K for TN paths, else K x N) and C."""
    g = si.generator(seed)
    dt = dtype(path)
    bshape = (N, K) if is_tn(path) else (K, N)
    if dist == "int":
        bound = 1 if dt != torch.float32 else 4
        A = si.small_integers((M, K), g, bound, dt)
        B = si.small_integers(bshape, g, bound, dt)
        C = si.small_integers((M, N), g, bound, dt)
    else:
        A, B, C = (si.uniform(sh, g).to(dt) for sh in ((M, K), bshape, (M, N)))
    if c_zero:
        C = torch.zeros_like(C)
    return A, B, C


def to_device_padded(t: torch.Tensor, pad: int = 0, fill=float("nan"), offset_elems: int = 0):
    """Copy a host matrix to the device inside a wider buffer (row pitch
    cols + pad, optional element offset of the base pointer); padding holds
    `fill` so that reads of it would show."""
    rows, cols = t.shape
    ld = cols + pad
    buf = torch.full((rows * ld + offset_elems + ld,), fill, dtype=t.dtype, device="cuda")
    view = buf[offset_elems:offset_elems + rows * ld].view(rows, ld)[:, :cols] if rows else \
        buf[:0].view(0, cols)
    view.copy_(t.to("cuda"))
    return view, buf


def run(path, A, B, C, alpha, beta, pad=(0, 0, 0), offset=(0, 0, 0), stream=None):
    """Run `path` on device copies of host A, B, C; returns (C_out host, C_dev_view, C_buf)."""
    dA, _ = to_device_padded(A, pad[0], offset_elems=offset[0])
    dB, _ = to_device_padded(B, pad[1], offset_elems=offset[1])
    dC, cbuf = to_device_padded(C, pad[2], fill=float("nan") if pad[2] else 0.0, offset_elems=offset[2])
    fn(path)(dA, dB, dC, alpha, beta, stream=stream)
    torch.cuda.synchronize()
    return dC.cpu(), dC, cbuf


def reference(path, A, B, C, alpha, beta, **select):
    return oracle.reference(oracle_kind(path), np_operand(A), np_operand(B), np_operand(C), alpha,
                            beta, tn=is_tn(path), **select)


def worst_ratio(path, got, A, B, C, alpha, beta, **select):
    """Max over the selected entries of |got - ref| / tolerance bound."""
    ref, ab = reference(path, A, B, C, alpha, beta, **select)
    K = A.shape[1]
    Cn = C.double().numpy()
    g = got.double().numpy() if isinstance(got, torch.Tensor) else got
    if "rows" in select:
        c_old = Cn[select["rows"]]
    elif "cols" in select:
        c_old = Cn[:, select["cols"]].T
    elif "entries" in select:
        c_old = Cn[select["entries"][0], select["entries"][1]]
    else:
        c_old = Cn
    r = oracle.violation_ratio(g, ref, ab, beta, c_old, tolerance(path, K))
    return float(r.max()) if r.size else 0.0


def sampled_check(path, got_dev: torch.Tensor, A, B, C, alpha, beta, n_samples=4096):
    """Large problems: 4096 seeded entries plus full rows and columns at tile
    boundaries.  Returns the worst ratio over all of them."""
    M, N = got_dev.shape
    K = A.shape[1]
    kind = oracle_kind(path)
    A64 = oracle.widen(kind, np_operand(A))
    B64 = oracle.widen(kind, np_operand(B), trans=is_tn(path))
    ck = kind if kind in ("f16", "bf16") else "f32"
    C64 = oracle.widen(ck, np_operand(C)) if beta != 0.0 else None
    Cd = C.double().numpy()
    ii, jj = si.sample_positions(M, N, n_samples)
    rows = si.boundary_indices(M)
    cols = si.boundary_indices(N)
    dev = got_dev.device
    tol = tolerance(path, K)
    worst = 0.0
    # rows
    got = got_dev[torch.as_tensor(rows, device=dev)].double().cpu().numpy()
    ref, ab = oracle.gemm(A64, B64, C64, alpha, beta, rows=rows)
    worst = max(worst, float(oracle.violation_ratio(got, ref, ab, beta, Cd[rows], tol).max()))
    # columns
    got = got_dev[:, torch.as_tensor(cols, device=dev)].T.contiguous().double().cpu().numpy()
    ref, ab = oracle.gemm(A64, B64, C64, alpha, beta, cols=cols)
    worst = max(worst, float(oracle.violation_ratio(got, ref, ab, beta, Cd[:, cols].T, tol).max()))
    # seeded entries
    got = got_dev[torch.as_tensor(ii, device=dev), torch.as_tensor(jj, device=dev)].double().cpu().numpy()
    ref, ab = oracle.gemm(A64, B64, C64, alpha, beta, entries=(ii, jj))
    worst = max(worst, float(oracle.violation_ratio(got, ref, ab, beta, Cd[ii, jj], tol).max()))
    return worst
