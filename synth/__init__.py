"""Seeded synthetic matrices shared by the tests, the bench and the oracle's callers.

This module holds no GEMM arithmetic. It only turns a counter-based random stream into
fp32 matrices of the shapes and value distributions of the SGEMM workloads:

* the stream is SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom
  number generators", OOPSLA 2014): output i of the stream seeded with ``s`` is
  ``mix(s + (i + 1) * 0x9E3779B97F4A7C15)`` modulo 2**64, where ``mix`` is the
  xor-shift-multiply finaliser with constants 0xBF58476D1CE4E5B9 and 0x94D049BB133111EB;
* element (r, c) of a ``rows x cols`` matrix takes counter ``r * cols + c`` (normal values take
  the counter pair ``2i, 2i + 1``), so a value depends only on its logical position, never on a
  leading dimension, and any row subset can be regenerated on its own;
* matrix A of a problem with seed ``s`` uses stream ``s``, B stream ``s + 1``, C stream ``s + 2``.

Distributions:
* ``uniform``: the top 24 bits give ``u`` in [0, 1) on a 2**-24 grid; the value is
  ``lo + (hi - lo) * u``. For [-1, 1) every value is exact in fp32.
* ``normal``: Box-Muller (G. Box, M. Muller, Ann. Math. Statist. 29, 1958) on two 53-bit
  uniforms, ``mu + sigma * sqrt(-2 ln u1) * cos(2 pi u2)`` in fp64, rounded once to fp32.
* ``small_int``: integers uniform in [lo, hi] (``(z >> 32) mod (hi - lo + 1)``), stored as fp32.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1
_CHUNK = 1 << 22  # counters per vectorised block (bounds temporary memory)


def splitmix64(seed: int, counters: np.ndarray) -> np.ndarray:
    """Outputs number ``counters`` (0-based, uint64) of the SplitMix64 stream seeded with ``seed``."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & _MASK64) + (c + np.uint64(1)) * GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
    return z ^ (z >> np.uint64(31))


def _rows_counters(row0: int, nrows: int, cols: int, per: int = 1) -> tuple[int, int]:
    start = row0 * cols * per
    return start, nrows * cols * per


def _fill(out_flat: np.ndarray, start: int, count: int, fn) -> None:
    for off in range(0, count, _CHUNK):
        n = min(_CHUNK, count - off)
        out_flat[off:off + n] = fn(np.arange(start + off, start + off + n, dtype=np.uint64))


def uniform(rows: int, cols: int, seed: int, lo: float = -1.0, hi: float = 1.0,
            row0: int = 0, nrows: int | None = None) -> np.ndarray:
    """Rows ``row0 .. row0 + nrows - 1`` of the ``rows x cols`` uniform [lo, hi) matrix."""
    nrows = rows - row0 if nrows is None else nrows
    out = np.empty((nrows, cols), dtype=np.float32)
    start, count = _rows_counters(row0, nrows, cols)

    def fn(idx):
        u = (splitmix64(seed, idx) >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
        return (lo + (hi - lo) * u).astype(np.float32)

    _fill(out.reshape(-1), start, count, fn)
    return out


def normal(rows: int, cols: int, seed: int, mu: float = 0.0, sigma: float = 1.0,
           row0: int = 0, nrows: int | None = None) -> np.ndarray:
    """Rows ``row0 .. row0 + nrows - 1`` of the ``rows x cols`` N(mu, sigma^2) matrix."""
    nrows = rows - row0 if nrows is None else nrows
    out = np.empty((nrows, cols), dtype=np.float32)
    start, count = _rows_counters(row0, nrows, cols)

    def fn(idx):
        z1 = splitmix64(seed, idx * np.uint64(2))
        z2 = splitmix64(seed, idx * np.uint64(2) + np.uint64(1))
        u1 = ((z1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
        u2 = (z2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)          # [0, 1)
        g = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        return (mu + sigma * g).astype(np.float32)

    _fill(out.reshape(-1), start, count, fn)
    return out


def small_int(rows: int, cols: int, seed: int, lo: int = -4, hi: int = 4,
              row0: int = 0, nrows: int | None = None) -> np.ndarray:
    """Rows of a ``rows x cols`` matrix of integers uniform in [lo, hi], stored as fp32."""
    nrows = rows - row0 if nrows is None else nrows
    out = np.empty((nrows, cols), dtype=np.float32)
    start, count = _rows_counters(row0, nrows, cols)
    span = np.uint64(hi - lo + 1)

    def fn(idx):
        v = ((splitmix64(seed, idx) >> np.uint64(32)) % span).astype(np.int64) + lo
        return v.astype(np.float32)

    _fill(out.reshape(-1), start, count, fn)
    return out


_DISTS = {"uniform": uniform, "normal": normal, "small_int": small_int}


def matrix(dist: str, rows: int, cols: int, seed: int, row0: int = 0,
           nrows: int | None = None, **params) -> np.ndarray:
    """Dispatch by distribution name: ``uniform`` (lo, hi), ``normal`` (mu, sigma), ``small_int``."""
    return _DISTS[dist](rows, cols, seed, row0=row0, nrows=nrows, **params)


def padded(mat: np.ndarray, ld: int, fill: float = np.nan) -> np.ndarray:
    """Copy a ``rows x cols`` matrix into a row-major buffer with leading dimension ``ld``.

    The padding columns hold ``fill`` (NaN by default) so that a read past the logical edge
    shows up in the result. Returns a ``rows x ld`` array.
    """
    rows, cols = mat.shape
    assert ld >= cols
    out = np.full((rows, ld), fill, dtype=np.float32)
    out[:, :cols] = mat
    return out
