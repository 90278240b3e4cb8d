"""The oracle's pins are sharp enough to catch plausible mistakes.

Each case plants one mistake in a temporary copy of the oracle's C source
(a transposed operand, a dropped term, a wrong sign, an off-by-one, a wrong
rounding or exponent bias), builds it with gcc on the CPU, swaps it in for
the real oracle and runs the pin suite: at least one pin must fail.
"""
import json
import os
import subprocess
import sys

import pytest

import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "dgemm_oracle.c")

MUTATIONS = {
    "transposed_operand_index": ("int64_t at = trans ? c * ld + r : r * ld + c;",
                                 "int64_t at = trans ? r * ld + c : c * ld + r;"),
    "dropped_beta_term": ("v += p->beta * p->C[i * N + j];\n        ref[j] = v;", "ref[j] = v;"),
    "wrong_sign_row_sum": ("ref[j] += a * brow[j];", "ref[j] -= a * brow[j];"),
    "k_off_by_one": ("for (int64_t k = 0; k < K; ++k) {\n            double a = p->A[i * K + k];\n            const",
                     "for (int64_t k = 0; k < K - 1; ++k) {\n            double a = p->A[i * K + k];\n            const"),
    "dropped_alpha": ("double v = (p->alpha != 0.0 && K > 0) ? p->alpha * ref[j] : 0.0;",
                      "double v = (p->alpha != 0.0 && K > 0) ? ref[j] : 0.0;"),
    "abs_without_fabs": ("abs_[j] += fabs(a) * fabs(brow[j]);", "abs_[j] += a * brow[j];"),
    "tf32_ties_to_even_instead_of_away": ("? trunc(n) : round(n);", "? trunc(n) : nearbyint(n);"),
    "tf32_keeps_11_bits": ("double q = ldexp(1.0, e - 10);", "double q = ldexp(1.0, e - 11);"),
    "tf32_no_subnormal_floor": ("if (e < -126)\n        e = -126;", "if (e < -160)\n        e = -160;"),
    "f16_bias_off_by_one": ("v = ldexp(1024.0 + (double)f, e - 25);", "v = ldexp(1024.0 + (double)f, e - 24);"),
    "f16_subnormal_scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "bf16_bias_off_by_one": ("v = ldexp(128.0 + (double)f, e - 134);", "v = ldexp(128.0 + (double)f, e - 133);"),
    "bf16_decoded_as_f16": ("v = oracle_bf16_value(((const uint16_t *)src)[at]);",
                            "v = oracle_f16_value(((const uint16_t *)src)[at]);"),
    "entry_uses_wrong_b_index": ("double b = p->B[k * N + j];", "double b = p->B[j * N + k];"),
    "beta_scales_the_sum_too": ("v += p->beta * p->C[i * N + j];\n        ref[j] = v;",
                                "v = p->beta * (v + p->C[i * N + j]);\n        ref[j] = v;"),
    "c_index_transposed": ("v += p->beta * p->C[i * N + j];\n    *ref = v;",
                           "v += p->beta * p->C[j * p->M + i];\n    *ref = v;"),
}

PIN_FUNCS = [
    ("test_hand_products", True), ("test_tf32_fixture", True), ("test_f16_fixture", True),
    ("test_bf16_fixture", True), ("test_bf16_all_patterns_match_torch", False),
    ("test_bf16_nn_and_tn_products_exact", False),
    ("test_f16_all_patterns_match_numpy", False),
    ("test_exact_integer_products", "kinds"), ("test_identity_and_permutation", "sizes"),
    ("test_rank_one_known_sums", False), ("test_alpha_zero_never_reads_operands", False),
    ("test_beta_zero_never_reads_c", False), ("test_k_zero_is_scaled_c", False),
    ("test_selection_modes_agree_with_full", False), ("test_tn_layout_is_transpose", False),
    ("test_tf32_kinds_round_operands_before_multiplying", False),
    ("test_tf32_matches_bit_definition", "modes"),
]


def _run_pins(golden_dir):
    failures = []
    for name, arg in PIN_FUNCS:
        fn = getattr(pins, name)
        calls = {True: [(golden_dir,)], False: [()],
                 "kinds": [("f32",), ("tf32_rna",), ("f16",)],
                 "sizes": [(5,), (33,)], "modes": [("tf32_rna",), ("tf32_rz",)]}[arg]
        for a in calls:
            try:
                fn(*a)
            except Exception as e:  # a pin that fails (or crashes) caught it
                failures.append((name, type(e).__name__))
    return failures


def _child(so_path, golden_dir):
    """Run the pins against the library at so_path (in a child process, so a
    mutant that crashes cannot take the test session with it)."""
    oracle._lib = oracle.load_library(so_path)
    print(json.dumps(_run_pins(golden_dir)))


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(mutation, tmp_path, golden_dir):
    old, new = MUTATIONS[mutation]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor not found: " + mutation
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-o", str(so), str(path), "-lm"])
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import sys; sys.path.insert(0, %r); import tests.test_oracle_mutations as m; "
            "m._child(%r, %r)" % (root, str(so), golden_dir))
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    if p.returncode < 0:
        return  # the mutant crashed (a signal) inside a pin: caught
    assert p.returncode == 0, p.stderr[-2000:]
    failures = json.loads(p.stdout.strip().splitlines()[-1])
    assert failures, "no pin caught the planted mistake " + mutation


def test_unmutated_oracle_passes_all_pins(golden_dir):
    assert _run_pins(golden_dir) == []
