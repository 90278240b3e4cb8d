"""Pins for the CPU oracle: it is checked against things other than itself.

Each test fixes the oracle to something the pages or the mathematics decide:
hand-computed products, closed forms (identity, permutation, rank-1,
alpha = 0, beta = 0), exact integer arithmetic, the operand formats'
definitions, and an independent library routine (numpy float64 matmul) on
small shapes.  The pins are chosen so that a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them.
"""
import json
import os
import struct

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si


def _f16(a):
    return np.asarray(a, dtype=np.float16)


# ---------------------------------------------------------------- golden ---

def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_hand_products(golden_dir):
    g = _golden(golden_dir, "hand_products.json")
    for case in g["cases"]:
        A = np.array(case["A"], dtype=np.float32)
        B = np.array(case["B"], dtype=np.float32)
        C = np.array(case["C"], dtype=np.float32)
        ref, ab = oracle.reference("f32", A, B, C, case["alpha"], case["beta"])
        assert np.array_equal(ref, np.array(case["ref"], dtype=np.float64)), case["name"]
        assert np.array_equal(ab, np.array(case["abs"], dtype=np.float64)), case["name"]
        # alpha = 1, beta = 0 gives the bare product
        ref1, _ = oracle.reference("f32", A, B, C, 1.0, 0.0)
        assert np.array_equal(ref1, np.array(case["AB"], dtype=np.float64))
        # the same numbers through every operand kind (all are exact here)
        for kind in ("tf32_rna", "tf32_rz"):
            r, _ = oracle.reference(kind, A, B, C, case["alpha"], case["beta"])
            assert np.array_equal(r, np.array(case["ref"], dtype=np.float64))
        if "B_tn_store" in case:
            Bt = _f16(case["B_tn_store"])
            r, a2 = oracle.reference("f16", _f16(case["A"]), Bt, _f16(case["C"]),
                                     case["alpha"], case["beta"], tn=True)
            assert np.array_equal(r, np.array(case["ref"], dtype=np.float64))
            assert np.array_equal(a2, np.array(case["abs"], dtype=np.float64))


def _hexf(s):
    return float(s) if s in ("inf", "-inf", "nan") else float.fromhex(s)


def test_tf32_fixture(golden_dir):
    g = _golden(golden_dir, "operand_values.json")
    for e in g["tf32"]:
        x = _hexf(e["x"])
        assert np.float32(x) == x, e  # the input is a float
        assert oracle.tf32_value(x, "tf32_rna") == _hexf(e["rna"]), e
        assert oracle.tf32_value(x, "tf32_rz") == _hexf(e["rz"]), e
        assert oracle.tf32_value(-x, "tf32_rna") == -_hexf(e["rna"]), e


def test_f16_fixture(golden_dir):
    g = _golden(golden_dir, "operand_values.json")
    for e in g["f16"]:
        v = oracle.f16_value(int(e["bits"], 16))
        want = _hexf(e["value"])
        if np.isnan(want):
            assert np.isnan(v)
        else:
            assert v == want and np.signbit(v) == np.signbit(want), e


def test_bf16_fixture(golden_dir):
    g = _golden(golden_dir, "operand_values.json")
    for e in g["bf16"]:
        v = oracle.bf16_value(int(e["bits"], 16))
        want = _hexf(e["value"])
        if np.isnan(want):
            assert np.isnan(v)
        else:
            assert v == want and np.signbit(v) == np.signbit(want), e


def test_bf16_all_patterns_match_torch():
    # every one of the 65536 bfloat16 patterns against torch's own decoder
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    mine = oracle.widen("bf16", bits)
    theirs = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).double().numpy()
    same = (mine == theirs) | (np.isnan(mine) & np.isnan(theirs))
    assert same.all()


def test_bf16_nn_and_tn_products_exact():
    # small integers are exact in bfloat16; NN reads B as K x N, TN as N x K
    g = si.generator(13)
    M, N, K = 9, 11, 40
    A = si.small_integers((M, K), g, dtype=torch.bfloat16)
    B = si.small_integers((K, N), g, dtype=torch.bfloat16)
    C = si.small_integers((M, N), g, dtype=torch.bfloat16)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    ref_nn, _ = oracle.reference("bf16", bits(A), bits(B), bits(C), 2.0, -1.0, tn=False)
    ref_tn, _ = oracle.reference("bf16", bits(A), bits(B.T), bits(C), 2.0, -1.0, tn=True)
    Ai, Bi, Ci = (t.to(torch.int64).numpy() for t in (A, B, C))
    want = (2 * (Ai @ Bi) - Ci).astype(np.float64)
    assert np.array_equal(ref_nn, want) and np.array_equal(ref_tn, want)


def test_f16_all_patterns_match_numpy():
    # every one of the 65536 binary16 patterns against numpy's own decoder
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    mine = oracle.widen("f16", bits)
    theirs = bits.view(np.float16).astype(np.float64)
    same = (mine == theirs) | (np.isnan(mine) & np.isnan(theirs))
    assert same.all()


def _tf32_bits(x32: np.ndarray, mode: str) -> np.ndarray:
    """TF32 from the bit layout: drop the 13 low fraction bits of the
    float32 pattern, after adding half of the dropped range for
    nearest-ties-away.  An independent statement of the same format."""
    u = x32.view(np.uint32).astype(np.uint64)
    if mode == "tf32_rna":
        u = u + 0x1000
    u = (u & 0xFFFFE000).astype(np.uint32)
    return u.view(np.float32).astype(np.float64)


@pytest.mark.parametrize("mode", ["tf32_rna", "tf32_rz"])
def test_tf32_matches_bit_definition(mode):
    rng = np.random.default_rng(7)
    pats = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    # keep finite patterns; add subnormals, ties and near-overflow patterns
    extra = np.array([0x00000001, 0x00001000, 0x00001FFF, 0x007FFFFF, 0x00800000,
                      0x3F801000, 0x3F803000, 0x3F800FFF, 0x7F7FFFFF, 0x7F7FEFFF,
                      0x80001000, 0xBF801000, 0x00002000, 0x00003000], dtype=np.uint32)
    pats = np.concatenate([pats, extra])
    x = pats.view(np.float32)
    x = x[np.isfinite(x)].reshape(1, -1)
    mine = oracle.widen(mode, x)[0]
    want = _tf32_bits(x[0].copy(), mode)
    assert np.array_equal(mine, want)


# ------------------------------------------------- numpy cross-check -------

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 9, 33), (64, 48, 80),
                                   (129, 127, 65), (256, 256, 256)])
def test_matches_numpy_float64(M, N, K):
    g = si.generator(M * 1000 + N * 10 + K)
    A, B, C = si.uniform((M, K), g).numpy(), si.uniform((K, N), g).numpy(), si.uniform((M, N), g).numpy()
    alpha, beta = 0.75, -1.25
    ref, ab = oracle.reference("f32", A, B, C, alpha, beta)
    A64, B64, C64 = A.astype(np.float64), B.astype(np.float64), C.astype(np.float64)
    want = alpha * (A64 @ B64) + beta * C64
    np.testing.assert_allclose(ref, want, rtol=1e-12, atol=1e-12 * K)
    np.testing.assert_allclose(ab, np.abs(A64) @ np.abs(B64), rtol=1e-12, atol=0)


def test_matches_numpy_512_cube():
    g = si.generator(512)
    A, B, C = (si.uniform((512, 512), g).numpy() for _ in range(3))
    ref, _ = oracle.reference("f32", A, B, C, 1.0, 0.5)
    want = A.astype(np.float64) @ B.astype(np.float64) + 0.5 * C.astype(np.float64)
    np.testing.assert_allclose(ref, want, rtol=1e-12, atol=1e-10)


def test_tn_layout_is_transpose():
    g = si.generator(3)
    M, N, K = 7, 11, 13
    A = si.uniform((M, K), g).half().numpy()
    Bt = si.uniform((N, K), g).half().numpy()   # TN store: N x K
    ref, _ = oracle.reference("f16", A, Bt, None, 1.0, 0.0, tn=True)
    want = A.astype(np.float64) @ Bt.astype(np.float64).T
    np.testing.assert_allclose(ref, want, rtol=1e-13, atol=1e-13)
    # the non-TN reading of the transposed copy gives the same product
    ref2, _ = oracle.reference("f16", A, np.ascontiguousarray(Bt.T), None, 1.0, 0.0, tn=False)
    assert np.array_equal(ref, ref2)


# ------------------------------------------------------- exact pins --------

@pytest.mark.parametrize("kind", ["f32", "tf32_rna", "tf32_rz", "f16"])
def test_exact_integer_products(kind):
    # small integers: every partial sum is an exact integer in double
    g = si.generator(11)
    M, N, K = 37, 41, 300
    dt = torch.float16 if kind == "f16" else torch.float32
    A = si.small_integers((M, K), g, dtype=dt).numpy()
    B = si.small_integers((K, N), g, dtype=dt).numpy()
    C = si.small_integers((M, N), g, dtype=dt).numpy()
    ref, ab = oracle.reference(kind, A, B, C, 1.0, 3.0)
    Ai, Bi, Ci = A.astype(np.int64), B.astype(np.int64), C.astype(np.int64)
    assert np.array_equal(ref, (Ai @ Bi + 3 * Ci).astype(np.float64))
    assert np.array_equal(ab, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))


def test_brute_force_python_integers():
    # pure-Python triple loop on a tiny non-square case, exact integers
    g = si.generator(5)
    M, N, K = 4, 6, 5
    A = si.small_integers((M, K), g).numpy()
    B = si.small_integers((K, N), g).numpy()
    C = si.small_integers((M, N), g).numpy()
    ref, _ = oracle.reference("f32", A, B, C, -2.0, 0.5)
    for i in range(M):
        for j in range(N):
            s = sum(int(A[i, k]) * int(B[k, j]) for k in range(K))
            assert ref[i, j] == -2.0 * s + 0.5 * float(C[i, j])


@pytest.mark.parametrize("M", [1, 5, 33])
def test_identity_and_permutation(M):
    g = si.generator(M)
    N = 9
    B = si.uniform((M, N), g).numpy()
    C = si.uniform((M, N), g).numpy()
    I = np.eye(M, dtype=np.float32)
    ref, _ = oracle.reference("f32", I, B, C, 1.0, 0.0)
    assert np.array_equal(ref, B.astype(np.float64))
    ref, _ = oracle.reference("f32", I, B, C, 1.0, 2.0)
    assert np.array_equal(ref, B.astype(np.float64) + 2.0 * C.astype(np.float64))
    perm = np.random.default_rng(M).permutation(M)
    P = np.zeros((M, M), dtype=np.float32)
    P[np.arange(M), perm] = 1.0
    ref, _ = oracle.reference("f32", P, B, C, 1.0, 0.0)
    assert np.array_equal(ref, B[perm].astype(np.float64))
    # TN: A = I gives C = B_store^T
    Bt = si.uniform((N, M), g).half().numpy()
    ref, _ = oracle.reference("f16", I.astype(np.float16), Bt, None, 1.0, 0.0, tn=True)
    assert np.array_equal(ref, Bt.T.astype(np.float64))


def test_rank_one_known_sums():
    M, N, K = 6, 7, 1000
    u = np.arange(1, M + 1, dtype=np.float32) * 0.5
    v = np.arange(-3, N - 3, dtype=np.float32)
    A = np.repeat(u[:, None], K, axis=1)
    B = np.repeat(v[None, :], K, axis=0)
    ref, _ = oracle.reference("f32", A, B, None, 1.0, 0.0)
    assert np.array_equal(ref, K * np.outer(u, v).astype(np.float64))
    # a = 1, b_kj = (k mod 8) - 4: the sum over k is an explicit integer
    A1 = np.ones((M, K), dtype=np.float32)
    Bk = np.repeat(((np.arange(K) % 8) - 4).astype(np.float32)[:, None], N, axis=1)
    ref, _ = oracle.reference("f32", A1, Bk, None, 1.0, 0.0)
    full, rem = divmod(K, 8)
    want = full * sum(r - 4 for r in range(8)) + sum(r - 4 for r in range(rem))
    assert np.all(ref == want)


def test_alpha_zero_never_reads_operands():
    M, N, K = 5, 6, 7
    A = np.full((M, K), np.nan, dtype=np.float32)
    B = np.full((K, N), np.nan, dtype=np.float32)
    C = np.arange(M * N, dtype=np.float32).reshape(M, N)
    ref, _ = oracle.reference("f32", A, B, C, 0.0, -1.5)
    assert np.array_equal(ref, -1.5 * C.astype(np.float64))
    ref, _ = oracle.reference("f32", A, B, C, 0.0, 0.0)
    assert np.array_equal(ref, np.zeros((M, N)))


def test_beta_zero_never_reads_c():
    g = si.generator(9)
    A, B = si.uniform((4, 3), g).numpy(), si.uniform((3, 5), g).numpy()
    C = np.full((4, 5), np.nan, dtype=np.float32)
    ref, _ = oracle.reference("f32", A, B, C, 1.0, 0.0)
    assert np.isfinite(ref).all()
    np.testing.assert_allclose(ref, A.astype(np.float64) @ B.astype(np.float64), rtol=1e-15)


def test_k_zero_is_scaled_c():
    C = np.array([[1.0, -2.0], [3.0, 0.5]], dtype=np.float32)
    A = np.zeros((2, 0), dtype=np.float32)
    B = np.zeros((0, 2), dtype=np.float32)
    ref, ab = oracle.reference("f32", A, B, C, 2.0, 3.0)
    assert np.array_equal(ref, 3.0 * C.astype(np.float64))
    assert np.array_equal(ab, np.zeros((2, 2)))


def test_a_zero_beta_nonzero_closed_form():
    g = si.generator(2)
    C = si.uniform((8, 8), g).numpy()
    A = np.zeros((8, 4), dtype=np.float32)
    B = si.uniform((4, 8), g).numpy()
    ref, _ = oracle.reference("f32", A, B, C, 1.0, 0.3)
    assert np.array_equal(ref, 0.3 * C.astype(np.float64))


# -------------------------------------------------- layout and modes -------

def test_padded_leading_dimensions_ignore_padding():
    g = si.generator(4)
    M, N, K = 9, 10, 11
    A = si.uniform((M, K), g).numpy()
    B = si.uniform((K, N), g).numpy()
    C = si.uniform((M, N), g).numpy()
    Ap = np.full((M, K + 5), np.nan, dtype=np.float32); Ap[:, :K] = A
    Bp = np.full((K, N + 3), np.nan, dtype=np.float32); Bp[:, :N] = B
    Cp = np.full((M, N + 32), np.nan, dtype=np.float32); Cp[:, :N] = C
    r1, a1 = oracle.reference("f32", A, B, C, 1.0, 1.0)
    r2, a2 = oracle.reference("f32", Ap[:, :K], Bp[:, :N], Cp[:, :N], 1.0, 1.0)
    assert np.array_equal(r1, r2) and np.array_equal(a1, a2)


def test_selection_modes_agree_with_full():
    g = si.generator(6)
    M, N, K = 130, 257, 33
    A, B, C = si.uniform((M, K), g).numpy(), si.uniform((K, N), g).numpy(), si.uniform((M, N), g).numpy()
    full, fabs_ = oracle.reference("f32", A, B, C, 1.5, -0.25)
    rows = si.boundary_indices(M)
    r, a = oracle.reference("f32", A, B, C, 1.5, -0.25, rows=rows)
    assert np.array_equal(r, full[rows]) and np.array_equal(a, fabs_[rows])
    cols = si.boundary_indices(N)
    r, a = oracle.reference("f32", A, B, C, 1.5, -0.25, cols=cols)
    assert np.array_equal(r, full[:, cols].T) and np.array_equal(a, fabs_[:, cols].T)
    ii, jj = si.sample_positions(M, N, 500)
    r, a = oracle.reference("f32", A, B, C, 1.5, -0.25, entries=(ii, jj))
    # entries use a dot product, rows an axpy sweep: same terms, same order
    assert np.array_equal(r, full[ii, jj]) and np.array_equal(a, fabs_[ii, jj])


def test_thread_count_does_not_change_results():
    g = si.generator(8)
    A, B = si.uniform((64, 50), g).numpy(), si.uniform((50, 70), g).numpy()
    r1, _ = oracle.reference("f32", A, B, None, 1.0, 0.0, nthreads=1)
    r7, _ = oracle.reference("f32", A, B, None, 1.0, 0.0, nthreads=7)
    assert np.array_equal(r1, r7)


def test_tf32_kinds_round_operands_before_multiplying():
    # a = 1 + 2^-11 (a TF32 tie), b = 1: the product shows the operand rounding
    A = np.array([[1.0 + 2.0 ** -11]], dtype=np.float32)
    B = np.array([[1.0]], dtype=np.float32)
    assert oracle.reference("f32", A, B, None, 1.0, 0.0)[0][0, 0] == 1.0 + 2.0 ** -11
    assert oracle.reference("tf32_rna", A, B, None, 1.0, 0.0)[0][0, 0] == 1.0 + 2.0 ** -10
    assert oracle.reference("tf32_rz", A, B, None, 1.0, 0.0)[0][0, 0] == 1.0
    # and B is rounded too (a transposed-operand or one-sided rounding slip fails)
    assert oracle.reference("tf32_rna", B, A, None, 1.0, 0.0)[0][0, 0] == 1.0 + 2.0 ** -10


# ------------------------------------------------------- acceptance rule ---

def test_violation_ratio():
    ref = np.array([1.0, 2.0, 0.0, 0.0])
    ab = np.array([1.0, 1.0, 0.0, 0.0])
    got = np.array([1.0 + 1e-4, 2.0 - 3e-3, 0.0, 1e-30])
    c = np.array([0.0, 4.0, 0.0, 0.0])
    r = oracle.violation_ratio(got, ref, ab, 0.5, c, 1e-3)
    assert r[0] == pytest.approx(0.1)
    assert r[1] == pytest.approx(3e-3 / (1e-3 + 2e-3))
    assert r[2] == 0.0 and r[3] == np.inf
