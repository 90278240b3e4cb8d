"""The C-ABI library builds, loads and exports every symbol include/dgemm.h
declares; host-side validation returns its status before touching a GPU.
No compute call is made here (these tests run without a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dgemm.h")


@pytest.fixture(scope="module")
def L():
    import dense_gemm_09_gb300 as dg
    dg.build()
    return dg.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ENTRY + ["dgemm_status_string", "dgemm_device_status"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    import dense_gemm_09_gb300 as dg
    out = subprocess.check_output(["nm", "-D", "--defined-only", dg.LIB_PATH], text=True)
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(L, name) is not None


def test_checked_build_exports_the_same_symbols(L):
    # the checked build (device-side bounds checks) has the same ABI
    import dense_gemm_09_gb300 as dg
    out = subprocess.check_output(["nm", "-D", "--defined-only", dg.LIB_CHECKED_PATH], text=True)
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
    Lc = dg.lib_checked()
    assert Lc.dgemm_test_shrink_bounds(-1) == 1   # DGEMM_ERR_INVALID_ARG
    assert Lc.dgemm_test_shrink_bounds(0) == 0


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "dgemm.h"\nint main(void){return gemm_f32(0,0,0,1.f,0,0,0,0,0.f,0,0,0);}\n')
    subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           "-c", str(src), "-o", str(tmp_path / "t.o")])


def test_status_strings(L):
    import dense_gemm_09_gb300 as dg
    for code in range(6):
        s = dg.status_string(code)
        assert s.startswith("DGEMM_"), s
    assert "unknown" in dg.status_string(99)


ENTRY = ["gemm_f32", "gemm_tf32", "gemm_f16_tn", "gemm_f16_nn", "gemm_bf16_tn", "gemm_bf16_nn"]
P = 0x1000  # a non-null dummy pointer value (never dereferenced: validation fails first)


@pytest.mark.parametrize("name", ENTRY)
@pytest.mark.parametrize("args", [
    (-1, 8, 8, 1.0, P, 8, P, 8, 0.0, P, 8),      # negative M
    (8, -1, 8, 1.0, P, 8, P, 8, 0.0, P, 8),      # negative N
    (8, 8, -1, 1.0, P, 8, P, 8, 0.0, P, 8),      # negative K
    (8, 8, 8, 1.0, P, 7, P, 8, 0.0, P, 8),       # lda < K
    (8, 8, 8, 1.0, P, 8, P, 7, 0.0, P, 8),       # ldb < row length of B
    (8, 8, 8, 1.0, P, 8, P, 8, 0.0, P, 7),       # ldc < N
    (8, 8, 8, 1.0, 0, 8, P, 8, 0.0, P, 8),       # A null but read
    (8, 8, 8, 1.0, P, 8, 0, 8, 0.0, P, 8),       # B null but read
    (8, 8, 8, 1.0, P, 8, P, 8, 0.0, 0, 8),       # C null
])
def test_invalid_arguments_rejected_on_host(L, name, args):
    st = getattr(L, name)(*args, None)
    assert st == 1  # DGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ENTRY)
def test_empty_problem_returns_ok_without_device(L, name):
    assert getattr(L, name)(0, 8, 8, 1.0, 0, 8, 0, 8, 0.0, 0, 8, None) == 0
    assert getattr(L, name)(8, 0, 8, 1.0, 0, 8, 0, 8, 0.0, 0, 8, None) == 0


@pytest.mark.parametrize("name", ENTRY)
def test_tn_ldb_rule(L, name):
    # TN: B is N x K, so ldb >= K is the rule (K=16 > N=8 here)
    st = getattr(L, name)(8, 8, 16, 1.0, P, 16, P, 8, 0.0, P, 8, None)
    if name.endswith("_tn"):
        assert st == 1
    else:
        assert st != 1  # ldb = N = 8 is valid for the NN calls


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a GPU")
@pytest.mark.parametrize("name", ENTRY)
def test_no_gpu_reports_unsupported_device(L, name):
    assert getattr(L, name)(8, 8, 8, 1.0, P, 8, P, 8, 0.0, P, 8, None) == 2


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import dense_gemm_09_gb300 as dg
    monkeypatch.setattr(dg, "_lib", None)
    monkeypatch.setattr(dg, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        dg.lib()


def test_last_kernel_empty_before_any_launch(L):
    assert L.dgemm_last_kernel() == b""


def test_tune_next_validates_on_host(L):
    # out-of-range requests are refused and record nothing (no device needed)
    assert L.dgemm_tune_next(-1, 256, 1) == 1
    assert L.dgemm_tune_next(9, 256, 1) == 1
    assert L.dgemm_tune_next(4, 256, 1) == 1     # 4 names no variant
    assert L.dgemm_tune_next(8, 192, 1) == 0     # the small-M pair: bn 128, 192 or 256
    assert L.dgemm_tune_next(8, 96, 1) == 1
    assert L.dgemm_tune_next(8, 160, 1) == 1
    assert L.dgemm_tune_next(6, 256, 2) == 0     # the finer-ring pair variants
    assert L.dgemm_tune_next(7, 256, 3) == 1     # (their split is a stream-K mode: 0..2)
    assert L.dgemm_tune_next(0, 0, 0) == 0
    assert L.dgemm_tune_next(2, 48, 1) == 1      # bn not a multiple of 32
    assert L.dgemm_tune_next(2, 288, 1) == 1     # bn above 256
    assert L.dgemm_tune_next(3, 128, 1) == 1     # split below 2
    assert L.dgemm_tune_next(3, 128, 9) == 1     # split above 8
    assert L.dgemm_tune_next(3, 128, 4) == 0
    assert L.dgemm_tune_next(5, 256, 3) == 1     # stream-K mode of a pair variant: 0..2
    assert L.dgemm_tune_next(1, 256, -1) == 1
    assert L.dgemm_tune_next(1, 256, 2) == 0
    assert L.dgemm_tune_next(0, 0, 0) == 0       # back to automatic


@pytest.mark.parametrize("args", [
    (-1, 8, 8, 1.0, P, 8, P, 8, 0.0, P, 8),      # negative M
    (8, 8, 8, 1.0, P, 7, P, 8, 0.0, P, 8),       # lda < K
    (8, 8, 8, 1.0, P, 8, P, 7, 0.0, P, 8),       # ldb < N
    (8, 8, 8, 1.0, P, 8, P, 8, 0.0, 0, 8),       # C null
])
def test_tf32_ws_invalid_arguments_rejected_on_host(L, args):
    assert L.gemm_tf32_ws(*args, P, 1 << 20, None) == 1
    assert L.gemm_f32_ws(*args, P, 1 << 20, None) == 1


def test_tf32_ws_empty_problem_returns_ok_without_device(L):
    assert L.gemm_tf32_ws(0, 8, 8, 1.0, 0, 8, 0, 8, 0.0, 0, 8, None, 0, None) == 0


def test_tf32_workspace_bytes_host_arithmetic(L):
    f = L.gemm_tf32_workspace_bytes
    # TMA-describable operands need no copy
    assert f(8192, 8192, 4096, P, 4096, P, 8192) == 0
    # the ragged workload (lda = 4095, ldb = 8193 floats): A as 8191 x 4096,
    # then B as 4095 x 8224 (whole 32-column groups) from the next 256-byte
    # boundary
    a = 8191 * 4096 * 4
    assert f(8191, 8193, 4095, P, 4095, P, 8193) == (a + 255) // 256 * 256 + 4095 * 8224 * 4
    # only A (base off a 16-byte boundary): 5 x 8 floats, padded to 256 bytes
    assert f(5, 8, 8, P + 4, 8, P, 8) == 256
    # only B (pitch of 9 floats): 8 x 32 floats
    assert f(5, 9, 8, P, 8, P, 9) == 8 * 32 * 4
    # K or M == 0: nothing to copy
    assert f(0, 9, 8, P + 4, 8, P, 9) == 0
    assert f(5, 9, 0, P + 4, 8, P, 9) == 0
    # invalid sizes, and copies past 2^63 bytes
    assert f(-1, 1, 1, P, 1, P, 1) == -1
    assert f(4, 4, 4, P, 3, P, 4) == -1
    assert f(2**40, 4, 2**30, P, 2**30 + 1, P, 4) == -1
