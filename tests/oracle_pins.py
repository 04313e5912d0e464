"""Pins for the CPU oracle: checks fixed by the definition of GEMM and by arithmetic,
not by the oracle itself. Each pin takes the oracle's ctypes handle, so the same checks
run against the real oracle (all must pass) and against deliberately broken copies of it
(each copy must fail at least one).

Sources of each pin:
* identity / permutation: A.I = A, I.B = B, P.B permutes rows of B, A.P permutes columns
  of A, exactly; the definition of each cell as a row-column dot product ("GEMM scrapbook",
  GEMM definition; "The 1% kernel", section 1).
* all-ones: a dot product of K ones with K ones is K.
* small integers: with |entries| <= 4 and K <= 16384 every partial sum is an integer below
  2**24, exact in any order, so the result equals the int64 product (numpy integer matmul,
  a separate routine) exactly.
* alpha/beta: C = alpha*(A.B) + beta*C ("a CUDA matmul", section 00) with the BLAS readings
  for beta = 0 (C not read), alpha = 0 (A, B not read) and K = 0.
* cancellation: terms exactly representable in fp32 whose running sum needs more than 24
  bits; the exact sum is representable, so one final rounding reproduces it.
* transposes: stored transposes through the ex entry agree with the plain product on
  numpy-transposed copies, with exact rational brute force, and with identity products.
* fused epilogue: each activation against its published formula evaluated with Python's
  math module; bias and residual against exact integer sums; activation before residual;
  the same on all four operand forms, with the operands stored transposed.
* denominators: sum_k |op(A)_ik| |op(B)_kj| on small integers equals numpy's int64 product of
  the absolute values of numpy-transposed copies, for all four operand forms.
* brute force: exact rational arithmetic (fractions.Fraction) on tiny shapes, rounded once
  to fp32; the oracle may differ by at most one fp32 ulp (its fp64 sum rounds before the
  final rounding).
"""
from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np

import oracle
import synth


def _mm(lib, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, rows=None):
    return oracle.sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, rows=rows, lib=lib)


def pin_identity(lib):
    for (M, K) in [(7, 7), (5, 9), (33, 17)]:
        A = synth.uniform(M, K, 11)
        eye = np.eye(K, dtype=np.float32)
        if not np.array_equal(_mm(lib, M, K, K, 1.0, A, K, eye, K, 0.0, None, K), A):
            return False
        B = synth.uniform(M, K, 12)  # M x K used as a K'=M rows matrix
        eyeM = np.eye(M, dtype=np.float32)
        if not np.array_equal(_mm(lib, M, K, M, 1.0, eyeM, M, B, K, 0.0, None, K), B):
            return False
    return True


def pin_permutation(lib):
    rng = np.random.default_rng(3)
    for (M, K, N) in [(6, 6, 6), (9, 5, 4), (4, 11, 13)]:
        p = rng.permutation(K)
        P = np.zeros((K, K), dtype=np.float32)
        P[np.arange(K), p] = 1.0                      # (P.B)[r] = B[p[r]]
        B = synth.uniform(K, N, 21)
        if not np.array_equal(_mm(lib, K, N, K, 1.0, P, K, B, N, 0.0, None, N), B[p]):
            return False
        A = synth.uniform(M, K, 22)
        # (A.P)[:, c] = sum_r A[:, r] P[r, c] = A[:, p^-1(c)]
        inv = np.argsort(p)
        if not np.array_equal(_mm(lib, M, K, K, 1.0, A, K, P, K, 0.0, None, K), A[:, inv]):
            return False
    return True


def pin_all_ones(lib):
    for (M, N, K) in [(3, 5, 1), (4, 3, 7), (2, 2, 4097), (3, 2, 16384)]:
        A = np.ones((M, K), dtype=np.float32)
        B = np.ones((K, N), dtype=np.float32)
        out = _mm(lib, M, N, K, 1.0, A, K, B, N, 0.0, None, N)
        if not np.array_equal(out, np.full((M, N), K, dtype=np.float32)):
            return False
    return True


def pin_small_int(lib):
    for (M, N, K, seed) in [(5, 7, 3, 0), (17, 13, 129, 1), (8, 9, 4099, 2), (3, 4, 16384, 3)]:
        A = synth.small_int(M, K, seed)
        B = synth.small_int(K, N, seed + 1)
        C = synth.small_int(M, N, seed + 2)
        exact = A.astype(np.int64) @ B.astype(np.int64)
        if not np.array_equal(_mm(lib, M, N, K, 1.0, A, K, B, N, 0.0, None, N),
                              exact.astype(np.float32)):
            return False
        # alpha = 2, beta = -3: still exact (|value| < 2**24)
        want = (2 * exact - 3 * C.astype(np.int64)).astype(np.float32)
        if not np.array_equal(_mm(lib, M, N, K, 2.0, A, K, B, N, -3.0, C, N), want):
            return False
    return True


def pin_alpha_beta(lib):
    M, N, K = 6, 5, 4
    A = synth.small_int(M, K, 5)
    B = synth.small_int(K, N, 6)
    C = synth.small_int(M, N, 7)
    S = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64)
    # beta = 0 ignores C, even NaN / Inf there
    Cbad = C.copy()
    Cbad[0, 0], Cbad[1, 1], Cbad[2, 3] = np.nan, np.inf, -np.inf
    out = _mm(lib, M, N, K, 1.5, A, K, B, N, 0.0, Cbad, N)
    if not np.array_equal(out, (1.5 * S).astype(np.float32)):
        return False
    # alpha = 0 ignores A and B, even NaN there
    Abad = A.copy()
    Abad[0, 0] = np.nan
    out = _mm(lib, M, N, K, 0.0, Abad, K, B, N, -0.5, C, N)
    if not np.array_equal(out, (-0.5 * C.astype(np.float64)).astype(np.float32)):
        return False
    # alpha = 0 and beta = 0 give zeros
    if not np.array_equal(_mm(lib, M, N, K, 0.0, Abad, K, B, N, 0.0, Cbad, N),
                          np.zeros((M, N), np.float32)):
        return False
    # K = 0 gives beta * C
    out = _mm(lib, M, N, 0, 1.0, np.zeros((M, 1), np.float32), 1, np.zeros((1, N), np.float32),
              N, 2.0, C, N)
    if not np.array_equal(out, (2.0 * C).astype(np.float32)):
        return False
    # alpha = 1, beta = 1: S + C
    out = _mm(lib, M, N, K, 1.0, A, K, B, N, 1.0, C, N)
    if not np.array_equal(out, (S + C).astype(np.float32)):
        return False
    # a NaN in A does reach the result when alpha != 0 (row 0 only)
    out = _mm(lib, M, N, K, 1.0, Abad, K, B, N, 0.0, None, N)
    if not (np.isnan(out[0]).all() and np.isfinite(out[1:]).all()):
        return False
    return True


def pin_cancellation(lib):
    # Exactly representable terms whose running sum needs more than 24 bits: the exact
    # result (1, 3, ...) is what "sum over k, then one rounding" gives; a sum kept in fp32
    # loses the small terms.
    big = float(2 ** 24)
    A = np.array([[big, 1.0, -big], [1.0, big, 3.0]], np.float32)
    B = np.array([[1.0], [1.0], [1.0]], np.float32)
    out = _mm(lib, 2, 1, 3, 1.0, A, 3, B, 1, 0.0, None, 1)
    want = np.array([[1.0], [big + 4.0]], np.float32)
    return np.array_equal(out, want)


def _exact_cell(A, B, C, i, j, alpha, beta):
    s = sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(A.shape[1]))
    v = Fraction(alpha) * s
    if beta != 0:
        v += Fraction(beta) * Fraction(float(C[i, j]))
    return v


def _ulp32(x: float) -> float:
    x = np.float32(abs(x))
    return float(np.spacing(x)) if x != 0 else float(np.finfo(np.float32).smallest_subnormal)


def pin_brute_force(lib):
    shapes = list(itertools.product([1, 2, 3, 5, 7], [1, 2, 4, 7], [1, 3, 6, 7]))
    for n, (M, N, K) in enumerate(shapes):
        A = synth.normal(M, K, 100 + n)
        B = synth.normal(K, N, 200 + n)
        C = synth.normal(M, N, 300 + n)
        alpha, beta = 0.7, -1.3
        out = _mm(lib, M, N, K, alpha, A, K, B, N, beta, C, N)
        for i in range(M):
            for j in range(N):
                exact = float(_exact_cell(A, B, C, i, j, alpha, beta))
                if abs(float(out[i, j]) - exact) > _ulp32(exact):
                    return False
    return True


def pin_leading_dims(lib):
    M, N, K = 9, 11, 13
    A = synth.normal(M, K, 31)
    B = synth.normal(K, N, 32)
    C = synth.normal(M, N, 33)
    packed = _mm(lib, M, N, K, 0.7, A, K, B, N, -1.3, C, N)
    Ap, Bp, Cp = synth.padded(A, K + 3), synth.padded(B, N + 5), synth.padded(C, N + 2)
    strided = _mm(lib, M, N, K, 0.7, Ap, K + 3, Bp, N + 5, -1.3, Cp, N + 2)
    return np.array_equal(packed, strided) and np.isfinite(strided).all()


def pin_row_subset(lib):
    M, N, K = 40, 23, 31
    A = synth.normal(M, K, 41)
    B = synth.normal(K, N, 42)
    C = synth.normal(M, N, 43)
    full = _mm(lib, M, N, K, 0.7, A, K, B, N, -1.3, C, N)
    rows = [39, 0, 17, 17, 5]
    sub = _mm(lib, M, N, K, 0.7, A, K, B, N, -1.3, C, N, rows=rows)
    return np.array_equal(sub, full[rows])


def _ex(lib, ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, rows=None):
    return oracle.sgemm_ex(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, rows=rows, lib=lib)


def pin_transposed_identity(lib):
    # I^T = I: op(A) = (A^T stored) with B = I gives back A, for every transpose flag.
    M, K = 9, 13
    A = synth.uniform(M, K, 61)
    At = np.ascontiguousarray(A.T)                # K x M storage of A^T
    eye = np.eye(K, dtype=np.float32)
    for tb in (False, True):
        if not np.array_equal(_ex(lib, True, tb, M, K, K, 1.0, At, M, eye, K, 0.0, None, K), A):
            return False
        if not np.array_equal(_ex(lib, False, tb, M, K, K, 1.0, A, K, eye, K, 0.0, None, K), A):
            return False
    return True


def pin_transposed_against_plain(lib):
    # op(A) op(B) on stored transposes equals the plain product on numpy-transposed copies
    # (numpy's transpose is a separate routine); padded leading dimensions included.
    M, N, K = 11, 7, 19
    A = synth.normal(M, K, 71)
    B = synth.normal(K, N, 72)
    C = synth.normal(M, N, 73)
    plain = _mm(lib, M, N, K, 0.7, A, K, B, N, -1.3, C, N)
    At = synth.padded(np.ascontiguousarray(A.T), M + 2)   # K x (M + 2)
    Bt = synth.padded(np.ascontiguousarray(B.T), K + 3)   # N x (K + 3)
    for ta, tb, a, lda, b, ldb in [(False, False, A, K, B, N), (True, False, At, M + 2, B, N),
                                   (False, True, A, K, Bt, K + 3), (True, True, At, M + 2, Bt, K + 3)]:
        got = _ex(lib, ta, tb, M, N, K, 0.7, a, lda, b, ldb, -1.3, C, N)
        if not np.array_equal(got, plain):
            return False
    return True


def pin_transposed_brute_force(lib):
    for n, (M, N, K) in enumerate([(1, 1, 1), (2, 3, 4), (5, 2, 3), (3, 7, 6)]):
        A = synth.normal(M, K, 400 + n)
        B = synth.normal(K, N, 500 + n)
        C = synth.normal(M, N, 600 + n)
        At, Bt = np.ascontiguousarray(A.T), np.ascontiguousarray(B.T)
        for ta in (False, True):
            for tb in (False, True):
                out = _ex(lib, ta, tb, M, N, K, 0.7, At if ta else A, M if ta else K,
                          Bt if tb else B, K if tb else N, -1.3, C, N)
                for i in range(M):
                    for j in range(N):
                        exact = float(_exact_cell(A, B, C, i, j, 0.7, -1.3))
                        if abs(float(out[i, j]) - exact) > _ulp32(exact):
                            return False
    return True


def pin_epilogue_activations(lib):
    # Pass chosen values x through the product (A = diag(x), B = I) and compare the fused
    # epilogue with each activation's formula evaluated by Python's math module, rounded to
    # fp32: a separate implementation of the published definitions.
    import math
    xs = np.array([-6.0, -2.5, -1.0, -0.25, 0.0, 0.5, 1.0, 3.0, 7.5], np.float32)
    n = len(xs)
    A = np.diag(xs).astype(np.float32)
    eye = np.eye(n, dtype=np.float32)
    forms = {
        "none": lambda x: x,
        "relu": lambda x: max(x, 0.0),
        "gelu": lambda x: 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0))),
        "gelu_tanh": lambda x: 0.5 * x * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) *
                                                          (x + 0.044715 * x ** 3))),
        "silu": lambda x: x / (1.0 + math.exp(-x)),
    }
    for act, f in forms.items():
        out = oracle.sgemm_epilogue(False, False, n, n, n, 1.0, A, n, eye, n, 0.0, None, n,
                                    None, act, lib=lib)
        want = np.diag([np.float32(f(float(x))) for x in xs])
        off = ~np.eye(n, dtype=bool)
        if not (np.array_equal(np.diag(out), np.diag(want)) and
                np.array_equal(out[off], np.full(off.sum(), np.float32(f(0.0))))):
            return False
    return True


def pin_epilogue_bias_and_residual(lib):
    # act = none: alpha * S + bias + beta * C on exact small integers equals the int64 sum.
    M, N, K = 7, 9, 33
    A, B, C = synth.small_int(M, K, 81), synth.small_int(K, N, 82), synth.small_int(M, N, 83)
    bias = synth.small_int(1, N, 84).reshape(-1)
    S = A.astype(np.int64) @ B.astype(np.int64)
    want = (2 * S + bias.astype(np.int64)[None, :] + 3 * C.astype(np.int64)).astype(np.float32)
    got = oracle.sgemm_epilogue(False, False, M, N, K, 2.0, A, K, B, N, 3.0, C, N, bias, "none",
                                lib=lib)
    if not np.array_equal(got, want):
        return False
    # relu is applied before the residual: relu(S + bias) + C
    want = (np.maximum(S + bias.astype(np.int64)[None, :], 0) + C.astype(np.int64)).astype(np.float32)
    got = oracle.sgemm_epilogue(False, False, M, N, K, 1.0, A, K, B, N, 1.0, C, N, bias, "relu",
                                lib=lib)
    return np.array_equal(got, want)


def _op_storage(X, trans, pad):
    """Storage of op(X) = X: X itself or its transpose, with `pad` columns of NaN padding."""
    s = np.ascontiguousarray(X.T) if trans else X
    ld = s.shape[1] + pad
    return synth.padded(s, ld, np.nan), ld


def pin_absdot(lib):
    # sum_k |op(A)_ik| |op(B)_kj| on small integers (all partial sums exact) against numpy's
    # int64 product of the absolute values; the stored operands carry padding between rows,
    # and A, B are not square, so a transposed index or a dropped absolute value shows.
    M, N, K = 7, 9, 33
    A = synth.small_int(M, K, 91)
    B = synth.small_int(K, N, 92)
    want = (np.abs(A).astype(np.int64) @ np.abs(B).astype(np.int64)).astype(np.float64)
    for ta in (False, True):
        for tb in (False, True):
            As, lda = _op_storage(A, ta, 3)
            Bs, ldb = _op_storage(B, tb, 2)
            As = np.where(np.isnan(As), 0.0, As).astype(np.float32)
            Bs = np.where(np.isnan(Bs), 0.0, Bs).astype(np.float32)
            got = oracle.absdot_ex(ta, tb, M, N, K, As, lda, Bs, ldb, lib=lib)
            if not np.array_equal(got, want):
                return False
            rows = [6, 0, 3]
            if not np.array_equal(oracle.absdot_ex(ta, tb, M, N, K, As, lda, Bs, ldb, rows=rows,
                                                   lib=lib), want[rows]):
                return False
    Ap, Bp = synth.padded(A, K + 3, 0.0), synth.padded(B, N + 2, 0.0)
    return np.array_equal(oracle.absdot(M, N, K, Ap, K + 3, Bp, N + 2, lib=lib), want)


def pin_epilogue_transposed(lib):
    # (1) act = none and relu on exact small integers, every operand form, stored transposes
    # with padding: act(2 S + bias) + 3 C equals the int64 value exactly.
    M, N, K = 6, 10, 21
    A, B, C = synth.small_int(M, K, 93), synth.small_int(K, N, 94), synth.small_int(M, N, 95)
    bias = synth.small_int(1, N, 96).reshape(-1)
    S = A.astype(np.int64) @ B.astype(np.int64)
    pre = 2 * S + bias.astype(np.int64)[None, :]
    for ta in (False, True):
        for tb in (False, True):
            As, lda = _op_storage(A, ta, 1)
            Bs, ldb = _op_storage(B, tb, 4)
            As = np.where(np.isnan(As), 0.0, As).astype(np.float32)
            Bs = np.where(np.isnan(Bs), 0.0, Bs).astype(np.float32)
            for act, f in (("none", lambda v: v), ("relu", lambda v: np.maximum(v, 0))):
                want = (f(pre) + 3 * C.astype(np.int64)).astype(np.float32)
                got = oracle.sgemm_epilogue(ta, tb, M, N, K, 2.0, As, lda, Bs, ldb, 3.0, C, N,
                                            bias, act, lib=lib)
                if not np.array_equal(got, want):
                    return False
    # (2) each activation through transposed storage: op(A) has the chosen values xs in its
    # first column and zeros elsewhere, op(B) ones in its first row, so every cell of row i
    # is act(xs[i]); compared with the formula evaluated by Python's math module.
    import math
    xs = np.array([-6.0, -2.5, -1.0, -0.25, 0.0, 0.5, 1.0, 3.0, 7.5], np.float32)
    n, Kx, Nx = len(xs), 3, 4
    A2 = np.zeros((n, Kx), np.float32)
    A2[:, 0] = xs
    B2 = np.zeros((Kx, Nx), np.float32)
    B2[0, :] = 1.0
    forms = {
        "gelu": lambda x: 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0))),
        "gelu_tanh": lambda x: 0.5 * x * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) *
                                                          (x + 0.044715 * x ** 3))),
        "silu": lambda x: x / (1.0 + math.exp(-x)),
    }
    for ta in (False, True):
        for tb in (False, True):
            As, lda = _op_storage(A2, ta, 2)
            Bs, ldb = _op_storage(B2, tb, 1)
            As = np.where(np.isnan(As), 0.0, As).astype(np.float32)
            Bs = np.where(np.isnan(Bs), 0.0, Bs).astype(np.float32)
            for act, f in forms.items():
                got = oracle.sgemm_epilogue(ta, tb, n, Nx, Kx, 1.0, As, lda, Bs, ldb, 0.0, None,
                                            Nx, None, act, lib=lib)
                want = np.array([[np.float32(f(float(x)))] * Nx for x in xs], np.float32)
                if not np.array_equal(got, want):
                    return False
    return True



def pin_page_counts(lib):
    """The counts the pages print for the 4096^3 problem (tests/golden/headline_counts.json):
    from the definition (2 n^3 FLOP, n^2 outputs, 3 n^2 four-byte inputs, their ratio), and
    through the oracle: an output cell sums exactly n products (A row and B all ones give
    C = n in every cell of the row), and one element of A reaches exactly n output cells (a
    single nonzero A[i0][k0] with B all ones fills row i0 and no other row)."""
    import json
    from pathlib import Path
    g = json.loads((Path(__file__).parent / "golden" / "headline_counts.json").read_text())
    n, pr = g["n"], g["printed"]
    ok = round(2 * n ** 3 / 1e9) == pr["flop_billions"]
    ok &= (n * n // 100_000) / 10 == pr["outputs_millions"]  # 16.78 million, printed cut to 16.7
    ok &= round(3 * n * n * 4 / 1e6) == pr["input_megabytes"]
    ok &= round(2 * n ** 3 / (3 * n * n * 4) / 10) * 10 == pr["flop_per_byte"]
    B = np.ones((n, n), np.float32)
    i0, k0, other = 1234, 777, 4095
    A = np.zeros((n, n), np.float32)
    A[i0, :] = 1.0
    rows = [i0, other]
    C = _mm(lib, n, n, n, 1.0, A, n, B, n, 0.0, None, n, rows=rows)
    ok &= bool(np.all(C[0] == pr["multiply_adds_per_output"]))
    ok &= bool(np.all(C[1] == 0.0))
    A[:] = 0.0
    A[i0, k0] = 1.0
    C = _mm(lib, n, n, n, 1.0, A, n, B, n, 0.0, None, n, rows=rows)
    ok &= int(np.count_nonzero(C[0])) == pr["output_cells_per_element_of_A"]
    ok &= int(np.count_nonzero(C[1])) == 0
    return bool(ok)

PINS = {
    "identity": pin_identity,
    "permutation": pin_permutation,
    "all_ones": pin_all_ones,
    "small_int": pin_small_int,
    "alpha_beta": pin_alpha_beta,
    "brute_force": pin_brute_force,
    "cancellation": pin_cancellation,
    "leading_dims": pin_leading_dims,
    "row_subset": pin_row_subset,
    "transposed_identity": pin_transposed_identity,
    "transposed_against_plain": pin_transposed_against_plain,
    "transposed_brute_force": pin_transposed_brute_force,
    "epilogue_activations": pin_epilogue_activations,
    "epilogue_bias_and_residual": pin_epilogue_bias_and_residual,
    "epilogue_transposed": pin_epilogue_transposed,
    "absdot": pin_absdot,
    "page_counts": pin_page_counts,
}
