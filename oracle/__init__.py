"""CPU oracle for C = alpha * (A . B) + beta * C on row-major fp32 matrices.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package. It shares no code with the CUDA library
(``dense_fp32_gemm_08_gb300``) and never imports it.

The arithmetic lives in ``sgemm_ref.c`` (plain C, fp64 accumulation in ascending k, one
rounding to fp32; the file's header lists the readings taken where the pages are silent).
This module only compiles that file with gcc, loads it with ctypes and marshals numpy
arrays. ``normalized_error`` is the acceptance metric applied to a GPU result.

Parity of real-valued outputs is pinned by invariants (identity, permutation, all-ones,
exact small-integer products, alpha/beta closed forms, brute force on tiny shapes), not by
worked values from the pages: the pages print none.
"""
from __future__ import annotations

import ctypes
import subprocess
import sys
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
SOURCE = _HERE / "sgemm_ref.c"
LIBRARY = _HERE / "liboracle_sgemm.so"

_lib = None


def build(source: Path = SOURCE, out: Path = LIBRARY, extra_flags: list[str] | None = None) -> Path:
    """Compile the C oracle into a shared library with gcc (OpenMP over result rows)."""
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-Wall", "-Wextra",
           str(source), "-o", str(out), "-lm"] + list(extra_flags or [])
    subprocess.run(cmd, check=True)
    return out


def _needs_build() -> bool:
    return (not LIBRARY.exists()) or LIBRARY.stat().st_mtime < SOURCE.stat().st_mtime


def load(path: Path | None = None):
    """Load (building first if missing or stale) and return the ctypes handle."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(str(path)))
    if _lib is None:
        if _needs_build():
            build()
        _lib = _bind(ctypes.CDLL(str(LIBRARY)))
    return _lib


def _bind(lib):
    i64, f64 = ctypes.c_int64, ctypes.c_double
    p = ctypes.c_void_p
    lib.sgemm_ref_rows.argtypes = [i64, i64, i64, f64, p, i64, p, i64, f64, p, i64, p, i64, p, i64]
    lib.sgemm_ref_rows.restype = ctypes.c_int
    lib.sgemm_ref_absdot_rows.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, p, i64]
    lib.sgemm_ref_absdot_rows.restype = ctypes.c_int
    i32 = ctypes.c_int
    lib.sgemm_ref_ex_rows.argtypes = [i32, i32, i64, i64, i64, f64, p, i64, p, i64, f64, p, i64,
                                      p, i64, p, i64]
    lib.sgemm_ref_ex_rows.restype = ctypes.c_int
    lib.sgemm_ref_absdot_ex_rows.argtypes = [i32, i32, i64, i64, i64, p, i64, p, i64, p, i64,
                                             p, i64]
    lib.sgemm_ref_absdot_ex_rows.restype = ctypes.c_int
    lib.sgemm_ref_epilogue_rows.argtypes = [i32, i32, i64, i64, i64, f64, p, i64, p, i64, f64, p,
                                            i64, p, i32, p, i64, p, i64]
    lib.sgemm_ref_epilogue_rows.restype = ctypes.c_int
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _as_f32(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.float32 or not a.flags.c_contiguous:
        raise TypeError("oracle inputs are C-contiguous float32 arrays")
    return a


def sgemm(M: int, N: int, K: int, alpha: float, A: np.ndarray, lda: int, B: np.ndarray, ldb: int,
          beta: float, C: np.ndarray | None, ldc: int, rows=None, lib=None) -> np.ndarray:
    """Result rows of C = alpha * A.B + beta * C (all M rows, or the listed ``rows``).

    ``A``, ``B``, ``C`` are flat or 2-D float32 buffers laid out row-major with the given
    leading dimensions; ``C`` may be None when ``beta == 0`` (and is then not read). Returns a float32 array of
    shape (len(rows) or M, N).
    """
    lib = lib or load()
    A = _as_f32(A)
    B = _as_f32(B)
    # C is handed over whenever the caller has one, so that "beta == 0 never reads C" is
    # something the oracle itself must honour (a NaN planted there must not surface).
    C = None if C is None else _as_f32(C)
    idx = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    R = M if idx is None else len(idx)
    out = np.empty((R, N), dtype=np.float32)
    st = lib.sgemm_ref_rows(M, N, K, float(alpha), _ptr(A), lda, _ptr(B), ldb, float(beta),
                            _ptr(C), ldc, _ptr(idx), 0 if idx is None else len(idx),
                            _ptr(out), max(N, 1))
    if st != 0:
        raise ValueError(f"oracle rejected the arguments (status {st})")
    return out


def sgemm_ex(transa: bool, transb: bool, M: int, N: int, K: int, alpha: float, A: np.ndarray,
             lda: int, B: np.ndarray, ldb: int, beta: float, C: np.ndarray | None, ldc: int,
             rows=None, lib=None) -> np.ndarray:
    """Like ``sgemm`` with transposed operands: A stored K x M when ``transa``, B stored
    N x K when ``transb`` (row-major, BLAS convention)."""
    lib = lib or load()
    A = _as_f32(A)
    B = _as_f32(B)
    C = None if C is None else _as_f32(C)
    idx = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    R = M if idx is None else len(idx)
    out = np.empty((R, N), dtype=np.float32)
    st = lib.sgemm_ref_ex_rows(int(bool(transa)), int(bool(transb)), M, N, K, float(alpha),
                               _ptr(A), lda, _ptr(B), ldb, float(beta), _ptr(C), ldc, _ptr(idx),
                               0 if idx is None else len(idx), _ptr(out), max(N, 1))
    if st != 0:
        raise ValueError(f"oracle rejected the arguments (status {st})")
    return out


ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2, "gelu_tanh": 3, "silu": 4}


def sgemm_epilogue(transa: bool, transb: bool, M: int, N: int, K: int, alpha: float,
                   A: np.ndarray, lda: int, B: np.ndarray, ldb: int, beta: float,
                   C: np.ndarray | None, ldc: int, bias: np.ndarray | None, act: str | int,
                   rows=None, lib=None) -> np.ndarray:
    """act(alpha * op(A) op(B) + bias) + beta * C, rounded once to fp32 (see sgemm_ref.c)."""
    lib = lib or load()
    A = _as_f32(A)
    B = _as_f32(B)
    C = None if C is None else _as_f32(C)
    bias = None if bias is None else _as_f32(np.ascontiguousarray(bias))
    code = ACTIVATIONS[act] if isinstance(act, str) else int(act)
    idx = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    R = M if idx is None else len(idx)
    out = np.empty((R, N), dtype=np.float32)
    st = lib.sgemm_ref_epilogue_rows(int(bool(transa)), int(bool(transb)), M, N, K, float(alpha),
                                     _ptr(A), lda, _ptr(B), ldb, float(beta), _ptr(C), ldc,
                                     _ptr(bias), code, _ptr(idx), 0 if idx is None else len(idx),
                                     _ptr(out), max(N, 1))
    if st != 0:
        raise ValueError(f"oracle rejected the arguments (status {st})")
    return out


def absdot_ex(transa: bool, transb: bool, M: int, N: int, K: int, A: np.ndarray, lda: int,
              B: np.ndarray, ldb: int, rows=None, lib=None) -> np.ndarray:
    """fp64 sum_k |op(A)[i][k]| * |op(B)[k][j]| for the listed rows."""
    lib = lib or load()
    A = _as_f32(A)
    B = _as_f32(B)
    idx = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    R = M if idx is None else len(idx)
    den = np.empty((R, N), dtype=np.float64)
    st = lib.sgemm_ref_absdot_ex_rows(int(bool(transa)), int(bool(transb)), M, N, K, _ptr(A),
                                      lda, _ptr(B), ldb, _ptr(idx),
                                      0 if idx is None else len(idx), _ptr(den), max(N, 1))
    if st != 0:
        raise ValueError(f"oracle rejected the arguments (status {st})")
    return den


def absdot(M: int, N: int, K: int, A: np.ndarray, lda: int, B: np.ndarray, ldb: int,
           rows=None, lib=None) -> np.ndarray:
    """fp64 sum_k |A[i][k]| * |B[k][j]| for the listed rows (all rows when ``rows`` is None)."""
    lib = lib or load()
    A = _as_f32(A)
    B = _as_f32(B)
    idx = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    R = M if idx is None else len(idx)
    den = np.empty((R, N), dtype=np.float64)
    st = lib.sgemm_ref_absdot_rows(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(idx),
                                   0 if idx is None else len(idx), _ptr(den), max(N, 1))
    if st != 0:
        raise ValueError(f"oracle rejected the arguments (status {st})")
    return den


def normalized_error(c_gpu: np.ndarray, c_ref: np.ndarray, absdot_ij: np.ndarray,
                     alpha: float, beta: float, c_in: np.ndarray | None) -> float:
    """max_ij |C_gpu - C_ref| / den_ij, taken with two denominators (the larger ratio wins).

    den1 = sum_k |A_ik||B_kj| + |beta| |C_ij|          (the acceptance formula as stated)
    den2 = |alpha| sum_k |A_ik||B_kj| + |beta| |C_ij|  (the same with alpha's scale)
    Where a denominator is zero the difference must be exactly zero (returns inf otherwise).
    NaN anywhere in the difference gives inf, unless both sides agree on NaN at that cell.
    """
    g = np.asarray(c_gpu, dtype=np.float64)
    r = np.asarray(c_ref, dtype=np.float64)
    both_nan = np.isnan(g) & np.isnan(r)
    same_inf = np.isinf(g) & np.isinf(r) & (np.sign(g) == np.sign(r))
    diff = np.where(both_nan | same_inf, 0.0, np.abs(g - r))
    if np.isnan(diff).any():
        return float("inf")
    cterm = 0.0 if (beta == 0.0 or c_in is None) else abs(beta) * np.abs(np.asarray(c_in, np.float64))
    worst = 0.0
    for den in (absdot_ij + cterm, abs(alpha) * absdot_ij + cterm):
        zero = den == 0.0
        if (diff[zero] != 0.0).any():
            return float("inf")
        if (~zero).any():
            worst = max(worst, float((diff[~zero] / den[~zero]).max()))
    return worst


def max_threads() -> int:
    return int(load().oracle_max_threads())


def set_threads(n: int) -> None:
    load().oracle_set_threads(int(n))


if __name__ == "__main__":  # `python -m oracle` builds the library
    print(build())
    sys.exit(0)
