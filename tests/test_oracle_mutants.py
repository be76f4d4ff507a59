"""Planted mistakes, on the CPU, in copies of the oracle: each mutant is
compiled from usm_oracle.c with one plausible error and must fail at least
one of the pins in test_oracle.py.  This shows the pins can see the mistakes
that matter (a wrong index, a dropped term, a transposed operand, a sign, a
reversed order, a wrong rounding tie)."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import workloads as W

SRC = os.path.join(os.path.dirname(oracle.__file__), "usm_oracle.c")

MUTANTS = {
    "spmm_row_for_col": ("const double *b = B + (int64_t)ci[p] * ldb;", "const double *b = B + (int64_t)r * ldb;"),
    "spmm_drop_last": ("for (int j = 0; j < N; ++j) c[j] += ap * b[j];",
                       "if (p + 1 < ro[r + 1]) for (int j = 0; j < N; ++j) c[j] += ap * b[j];"),
    "sddmm_operand_not_transposed": ("for (int j = 0; j < D; ++j) s += x[j] * y[j];",
                                     "for (int j = 0; j < D; ++j) s += x[j] * Y[(int64_t)j * ldy + ci[p]];"),
    "sddmm_sign": ("out[p] = s;\n", "out[p] = -s;\n"),
    "swizzle_ties_reversed": ("return a < b ? -1 : (a > b ? 1 : 0);", "return a < b ? 1 : (a > b ? -1 : 0);"),
    "swizzle_ascending": ("if (la != lb) return la > lb ? -1 : 1;", "if (la != lb) return la < lb ? -1 : 1;"),
    "transpose_wrong_index": ("ci_t[q] = r;", "ci_t[q] = c;"),
    "softmax_no_shift_in_sum": ("for (int32_t p = b; p < e; ++p) z += exp(s[p] - m);",
                                "for (int32_t p = b; p < e; ++p) z += exp(s[p]);"),
    "bf16_ties_away": ("if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;",
                       "if (rem >= 0.5) fl += 1.0;"),
    # CSR contract check.  (Dropping the row_offsets[M] = nnz rule is left
    # out: the mutant would then read past the end of col_indices.)
    "csr_check_allows_duplicates": ("if (p > ro[r] && ci[p] <= ci[p - 1]) return -6;",
                                    "if (p > ro[r] && ci[p] < ci[p - 1]) return -6;"),
    "csr_check_allows_K": ("if (ci[p] < 0 || ci[p] >= K) return -5;", "if (ci[p] < 0 || ci[p] > K) return -5;"),
    "csr_check_ignores_decrease": ("if (ro[r + 1] < ro[r]) return -3;", "if (ro[r + 1] < ro[r] - 1000000) return -3;"),
}


def build_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC", "-std=c11",
                    str(path), "-o", str(so), "-lm"], check=True)
    return oracle._configure(ctypes.CDLL(str(so)))


def pins_pass(golden_dir):
    """Run a compact version of the pins; True when all hold."""
    import test_oracle as T
    checks = [
        lambda: T.test_golden_spmm(golden_dir),
        lambda: T.test_golden_sddmm(golden_dir),
        lambda: T.test_golden_swizzle(golden_dir),
        lambda: T.test_golden_transpose(golden_dir),
        lambda: T.test_golden_bf16_rounding(golden_dir),
        lambda: T.test_golden_softmax(golden_dir),
        lambda: T.test_spmm_vs_dense(33, 17, 9, 0.3),
        lambda: T.test_sddmm_vs_dense_masked(64, 64, 64, 0.3),
        lambda: T.test_swizzle_vs_lexsort(1000, 300, 0),
        lambda: T.test_transpose_vs_dense(20, 30, 0.2),
        lambda: T.test_csr_check_rejects_corruption(),
    ]
    for c in checks:
        try:
            c()
        except AssertionError:
            return False
    return True


def test_pins_pass_on_real_oracle(golden_dir):
    assert pins_pass(golden_dir)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, golden_dir, monkeypatch):
    lib = build_mutant(name, tmp_path)
    monkeypatch.setattr(oracle, "_lib", lib)
    assert not pins_pass(golden_dir), f"planted mistake {name} went unnoticed"
