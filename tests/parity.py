"""Helpers for the GPU parity tests: run a path through the C ABI binding on
seeded host operands and compare with the CPU oracle element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import seeded_inputs as si

PATHS = ("f32", "tf32", "f16_tn")


def tolerance(path: str, K: int) -> float:
    return {"f32": oracle.tol_f32(K), "tf32": oracle.TOL_TF32, "f16_tn": oracle.TOL_F16}[path]


def oracle_kind(path: str) -> str:
    # TF32: the kernel feeds the stored FP32 operands to the tensor core,
    # which keeps their top 19 bits (truncation toward zero, measured with
    # crafted operands -- see test_tf32_operand_rounding_is_truncation); the
    # oracle reduces operands the same way.
    return {"f32": "f32", "tf32": "tf32_rz", "f16_tn": "f16"}[path]


def host_operands(path, M, N, K, seed=0, dist="uniform", c_zero=False):
    g = si.generator(seed)
    if path == "f16_tn":
        if dist == "int":
            A = si.small_integers((M, K), g, 1, torch.float16)
            B = si.small_integers((N, K), g, 1, torch.float16)
            C = si.small_integers((M, N), g, 1, torch.float16)
        else:
            A, B = si.uniform((M, K), g).half(), si.uniform((N, K), g).half()
            C = si.uniform((M, N), g).half()
    else:
        if dist == "int":
            A = si.small_integers((M, K), g, 4)
            B = si.small_integers((K, N), g, 4)
            C = si.small_integers((M, N), g, 4)
        else:
            A, B, C = si.uniform((M, K), g), si.uniform((K, N), g), si.uniform((M, N), g)
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
    import dense_gemm_09_gb300 as dg
    dA, _ = to_device_padded(A, pad[0], offset_elems=offset[0])
    dB, _ = to_device_padded(B, pad[1], offset_elems=offset[1])
    dC, cbuf = to_device_padded(C, pad[2], fill=float("nan") if pad[2] else 0.0, offset_elems=offset[2])
    fn = {"f32": dg.gemm_f32, "tf32": dg.gemm_tf32, "f16_tn": dg.gemm_f16_tn}[path]
    fn(dA, dB, dC, alpha, beta, stream=stream)
    torch.cuda.synchronize()
    return dC.cpu(), dC, cbuf


def reference(path, A, B, C, alpha, beta, **select):
    return oracle.reference(oracle_kind(path), A.numpy(), B.numpy(), C.numpy(), alpha, beta,
                            tn=(path == "f16_tn"), **select)


def worst_ratio(path, got, A, B, C, alpha, beta, **select):
    """Max over the selected entries of |got - ref| / tolerance bound."""
    ref, ab = reference(path, A, B, C, alpha, beta, **select)
    K = A.shape[1]
    Cn = C.numpy().astype(np.float64)
    g = got.numpy() if isinstance(got, torch.Tensor) else got
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
    A64 = oracle.widen(kind, A.numpy())
    B64 = oracle.widen(kind, B.numpy(), trans=(path == "f16_tn"))
    Cn = C.numpy()
    C64 = oracle.widen("f16" if path == "f16_tn" else "f32", Cn) if beta != 0.0 else None
    Cd = Cn.astype(np.float64)
    ii, jj = si.sample_positions(M, N, n_samples)
    rows = si.boundary_indices(M)
    cols = si.boundary_indices(N)
    dev = got_dev.device
    tol = tolerance(path, K)
    worst = 0.0
    # rows
    got = got_dev[torch.as_tensor(rows, device=dev)].cpu().numpy()
    ref, ab = oracle.gemm(A64, B64, C64, alpha, beta, rows=rows)
    worst = max(worst, float(oracle.violation_ratio(got, ref, ab, beta, Cd[rows], tol).max()))
    # columns
    got = got_dev[:, torch.as_tensor(cols, device=dev)].T.contiguous().cpu().numpy()
    ref, ab = oracle.gemm(A64, B64, C64, alpha, beta, cols=cols)
    worst = max(worst, float(oracle.violation_ratio(got, ref, ab, beta, Cd[:, cols].T, tol).max()))
    # seeded entries
    got = got_dev[torch.as_tensor(ii, device=dev), torch.as_tensor(jj, device=dev)].cpu().numpy()
    ref, ab = oracle.gemm(A64, B64, C64, alpha, beta, entries=(ii, jj))
    worst = max(worst, float(oracle.violation_ratio(got, ref, ab, beta, Cd[ii, jj], tol).max()))
    return worst
