"""Planted mistakes: each is applied to a copy of the oracle's C source,
compiled on the CPU, and must make at least one pin fail.  This shows that
the pins would notice a dropped term, a wrong sign, a wrong index or leading
dimension, a transposed operand or a lost bit of precision in the oracle."""
import os

import pytest

import oracle
from tests.oracle_pins import PINS

MUTANTS = {
    "drop_last_k_term": ("acc[j] += a * (double)Bp[j];",
                         "acc[j] += (p + 1 < K) ? a * (double)Bp[j] : 0.0;"),
    "beta_sign": ("acc[j] = acc[j] + beta * (double)c0[j];",
                  "acc[j] = acc[j] - beta * (double)c0[j];"),
    "drop_alpha": ("acc[j] = alpha * acc[j];", "acc[j] = acc[j];"),
    "read_c_when_beta_zero": ("if (beta != 0.0) {", "if (1) {"),
    "read_ab_when_alpha_zero": ("if (alpha != 0.0 && K > 0) {", "if (K > 0) {"),
    "b_rows_at_n_not_ldb": ("const float *Bp = B + (int64_t)p * ldb;",
                            "const float *Bp = B + (int64_t)p * N;"),
    "a_row_offset_without_lda": (
        "row_f64(N, K, (double)alpha, A + (int64_t)i * lda, B, ldb,\n                    (double)beta, Ci, acc);",
        "row_f64(N, K, (double)alpha, A + (int64_t)i, B, ldb,\n                    (double)beta, Ci, acc);"),
    "b_transposed": ("acc[j] += a * (double)Bp[j];",
                     "acc[j] += a * (double)B[((int64_t)j * ldb + p) % ((int64_t)K * ldb)];"),
    "accumulate_in_float": ("acc[j] += a * (double)Bp[j];",
                            "acc[j] = (float)(acc[j] + a * (double)Bp[j]);"),
    "last_column_skipped": ("for (int j = 0; j < N; ++j)\n                acc[j] += a",
                            "for (int j = 0; j < N - 1; ++j)\n                acc[j] += a"),
    "round_twice": ("acc[j] = alpha * acc[j];", "acc[j] = (float)(alpha * (float)acc[j]);"),
}


def _source_with(old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    return src.replace(old, new, 1)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = tmp_path / "mutant.c"
    src.write_text(_source_with(old, new))
    so = oracle.compile_oracle(str(src), str(tmp_path / "libmutant.so"))
    lib = oracle.load_library(so)
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
