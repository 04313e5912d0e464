"""The oracle against checks that the definition of GEMM and plain arithmetic fix, and
the same checks against broken copies of the oracle (each must be caught)."""
from __future__ import annotations

import subprocess
import sys
from pathlib import Path

import numpy as np
import pytest

import oracle
import synth
from oracle_pins import PINS


@pytest.mark.parametrize("name", sorted(PINS))
def test_pin(name, oracle_lib):
    assert PINS[name](oracle_lib), f"oracle fails pin {name}"


# Plausible mistakes, planted in a copy of the oracle's C source (never in the tree).
# Each entry: (text in sgemm_ref.c, replacement).
MUTANTS = {
    "dropped_beta_term": ("if (beta != 0.0) v += beta * (double)C[i * ldc + j];",
                          "(void)beta;"),
    "transposed_B": ("    s.bk = transb ? 1 : ldb;\n    s.bj = transb ? ldb : 1;",
                     "    s.bk = transb ? ldb : 1;\n    s.bj = transb ? 1 : ldb;"),
    "transposed_A": ("    s.ai = transa ? 1 : lda;\n    s.ak = transa ? lda : 1;",
                     "    s.ai = transa ? lda : 1;\n    s.ak = transa ? 1 : lda;"),
    "dropped_last_k": ("for (int64_t k = 0; k < K; ++k) {\n                    const double a = (double)A",
                       "for (int64_t k = 0; k + 1 < K; ++k) {\n                    const double a = (double)A"),
    "alpha_sign": ("double v = (alpha != 0.0) ? alpha * acc[j] : 0.0;",
                   "double v = (alpha != 0.0) ? -alpha * acc[j] : 0.0;"),
    "beta_zero_reads_C": ("if (beta != 0.0) v += beta * (double)C[i * ldc + j];",
                          "v += beta * (double)C[i * ldc + j];"),
    "fp32_accumulator": ("acc[j] += a * (double)brow[j * st.bj];",
                         "acc[j] = (double)((float)acc[j] + (float)(a * (double)brow[j * st.bj]));"),
    "alpha_scales_C": ("if (beta != 0.0) v += beta * (double)C[i * ldc + j];",
                       "if (beta != 0.0) v += alpha * beta * (double)C[i * ldc + j];"),
    "ldc_ignored": ("if (beta != 0.0) v += beta * (double)C[i * ldc + j];",
                    "if (beta != 0.0) v += beta * (double)C[i * N + j];"),
    "lda_for_ldb": ("    s.bk = transb ? 1 : ldb;", "    s.bk = transb ? 1 : lda;"),
    "ex_transposed_A_index": ("    s.ai = transa ? 1 : lda;\n    s.ak = transa ? lda : 1;",
                              "    s.ai = lda;\n    s.ak = 1;"),
    "ex_transposed_B_index": ("    s.bk = transb ? 1 : ldb;\n    s.bj = transb ? ldb : 1;",
                              "    s.bk = ldb;\n    s.bj = 1;"),
    "ex_ignores_transpose": ("return product_rows(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, NULL, 0,",
                             "return product_rows(0, 0, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, NULL, 0,"),
    "epilogue_ignores_transpose": ("return product_rows(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias, act,",
                                   "return product_rows(0, 0, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias, act,"),
    "epilogue_gelu_constant": ("return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));",
                               "return 0.5 * x * (1.0 + erf(x / 2.0));"),
    "epilogue_act_after_residual": ("                v = activation(v, act);\n                if (beta != 0.0) v += beta * (double)C[i * ldc + j];",
                                    "                if (beta != 0.0) v += beta * (double)C[i * ldc + j];\n                v = activation(v, act);"),
    "epilogue_bias_dropped": ("if (bias) v += (double)bias[j];", "(void)bias;"),
    "wrong_row_index": ("const int64_t i = rows ? rows[r] : r;\n            for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;",
                        "const int64_t i = r;\n            for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;"),
    "absdot_dropped_abs_A": ("const double a = fabs((double)A[i * st.ai + k * st.ak]);",
                             "const double a = (double)A[i * st.ai + k * st.ak];"),
    "absdot_dropped_abs_B": ("drow[j] += a * fabs((double)brow[j * st.bj]);",
                             "drow[j] += a * (double)brow[j * st.bj];"),
    "absdot_ignores_transpose": ("    const op_strides st = strides_of(transa, transb, lda, ldb);\n#pragma omp parallel for",
                                 "    const op_strides st = strides_of(0, 0, lda, ldb);\n#pragma omp parallel for"),
    "absdot_wrong_row_index": ("const int64_t i = rows ? rows[r] : r;\n        double *drow",
                               "const int64_t i = r;\n        double *drow"),
    "absdot_plain_transposes": ("return sgemm_ref_absdot_ex_rows(0, 0, M,",
                                "return sgemm_ref_absdot_ex_rows(0, 1, M,"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("mutants")


_CHILD = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle
from oracle_pins import PINS
lib = oracle.load({lib!r})
failed = []
for name, fn in PINS.items():
    try:
        ok = fn(lib)
    except Exception:
        ok = False
    if not ok:
        failed.append(name)
print("FAILED_PINS", ",".join(failed))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, mutant_dir):
    src = oracle.SOURCE.read_text()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} must occur exactly once"
    path = mutant_dir / f"{name}.c"
    path.write_text(src.replace(old, new, 1))
    lib_path = oracle.build(path, mutant_dir / f"lib{name}.so")
    tests_dir = Path(__file__).resolve().parent
    code = _CHILD.format(root=str(tests_dir.parent), tests=str(tests_dir), lib=str(lib_path))
    # A child process: a mutant that reads out of bounds may crash, and a crash is a catch.
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                          timeout=600)
    if proc.returncode != 0:
        return
    line = [l for l in proc.stdout.splitlines() if l.startswith("FAILED_PINS")][-1]
    caught = [x for x in line.split(" ", 1)[1].split(",") if x]
    assert caught, f"no pin catches the planted mistake {name}"


def test_normalized_error_metric():
    # A planted error of known size gives the expected ratio with both denominators.
    ref = np.array([[1.0, -2.0]], np.float32)
    den = np.array([[4.0, 8.0]])
    got = ref.copy()
    got[0, 1] += 0.5
    e = oracle.normalized_error(got, ref, den, alpha=0.5, beta=0.0, c_in=None)
    assert e == pytest.approx(0.5 / 4.0)  # |alpha| * 8 = 4 is the smaller denominator
    assert oracle.normalized_error(ref, ref, den, 1.0, 0.0, None) == 0.0
    # zero denominator: any difference is infinite error, no difference is fine
    zden = np.zeros((1, 2))
    assert oracle.normalized_error(ref, ref, zden, 1.0, 0.0, None) == 0.0
    assert oracle.normalized_error(got, ref, zden, 1.0, 0.0, None) == float("inf")
    # NaN on one side only is an error; on both sides it is agreement
    nan_ref = ref.copy()
    nan_ref[0, 0] = np.nan
    assert oracle.normalized_error(ref, nan_ref, den, 1.0, 0.0, None) == float("inf")
    assert oracle.normalized_error(nan_ref, nan_ref, den, 1.0, 0.0, None) == 0.0
    # the beta term joins the denominator
    cin = np.array([[10.0, 10.0]], np.float32)
    e = oracle.normalized_error(got, ref, den, 1.0, 2.0, cin)
    assert e == pytest.approx(0.5 / (8.0 + 20.0))


def test_absdot_closed_form(oracle_lib):
    M, N, K = 7, 9, 33
    A = synth.small_int(M, K, 51)
    B = synth.small_int(K, N, 52)
    den = oracle.absdot(M, N, K, A, K, B, N, lib=oracle_lib)
    want = np.abs(A).astype(np.int64) @ np.abs(B).astype(np.int64)
    assert np.array_equal(den, want.astype(np.float64))
    # on non-negative inputs the denominator equals the product itself
    Ap, Bp = np.abs(A), np.abs(B)
    assert np.array_equal(oracle.sgemm(M, N, K, 1.0, Ap, K, Bp, N, 0.0, None, N).astype(np.float64),
                          oracle.absdot(M, N, K, Ap, K, Bp, N))


def test_argument_rejection(oracle_lib):
    A = np.zeros((2, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.sgemm(-1, 2, 2, 1.0, A, 2, A, 2, 0.0, None, 2)
    with pytest.raises(ValueError):
        oracle.sgemm(2, 2, 2, 1.0, A, 1, A, 2, 0.0, None, 2)  # lda < K
    with pytest.raises(ValueError):
        oracle.sgemm(2, 2, 2, 1.0, A, 2, A, 2, 0.0, None, 2, rows=[2])  # row out of range


def test_page_counts():
    # The exact values behind the pages' rounded counts (tests/golden/headline_counts.json,
    # whose printed figures the oracle pin "page_counts" checks).
    n = 4096
    assert 2 * n ** 3 == 137_438_953_472
    assert n * n == 16_777_216
    assert 3 * n * n * 4 == 201_326_592
