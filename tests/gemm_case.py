"""Shared driver for GPU-versus-oracle cases: builds seeded inputs, places them in device
buffers with optional padding, pointer offsets and guard bands, runs one library entry point
through the C ABI, and compares the result with the oracle."""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

import oracle
import synth

TOL = 1e-5           # normalised-error bound for fp32 results (all paths)
SENTINEL = 12345.5   # value kept in C's padding and guard band; must survive every call
GUARD = 64           # floats of guard band after each device buffer


@dataclass
class Case:
    M: int
    N: int
    K: int
    alpha: float = 1.0
    beta: float = 0.0
    dist: str = "uniform"              # uniform | normal | small_int | llm
    seed: int = 0
    lda_pad: int = 0
    ldb_pad: int = 0
    ldc_pad: int = 0
    a_off: int = 0                     # pointer offsets in floats (misalignment)
    b_off: int = 0
    c_off: int = 0
    rows: list | None = None           # result rows to check (None = all)
    nan_c_when_beta0: bool = False     # plant NaN/Inf in C (must not reach the result)
    extra: dict = field(default_factory=dict)

    @property
    def lda(self):
        return max(self.K, 1) + self.lda_pad

    @property
    def ldb(self):
        return max(self.N, 1) + self.ldb_pad

    @property
    def ldc(self):
        return max(self.N, 1) + self.ldc_pad


def inputs(case: Case, rows_a=None):
    """Host matrices A (M x K), B (K x N), C (M x N) for the case's distribution."""
    M, N, K, s = case.M, case.N, case.K, case.seed
    if case.dist == "uniform":
        A, B, C = synth.uniform(M, K, s), synth.uniform(K, N, s + 1), synth.uniform(M, N, s + 2)
    elif case.dist == "normal":
        A, B, C = synth.normal(M, K, s), synth.normal(K, N, s + 1), synth.normal(M, N, s + 2)
    elif case.dist == "small_int":
        A, B, C = synth.small_int(M, K, s), synth.small_int(K, N, s + 1), synth.small_int(M, N, s + 2)
    elif case.dist == "llm":
        A = synth.normal(M, K, s)
        B = synth.normal(K, N, s + 1, sigma=0.02)
        C = synth.normal(M, N, s + 2)
    else:
        raise ValueError(case.dist)
    if case.nan_c_when_beta0 and M > 0 and N > 0:
        C = C.copy()
        C[0, 0] = np.nan
        C[M - 1, N - 1] = np.inf
        C[M // 2, N // 2] = -np.inf
    return A, B, C


def to_device(torch, host: np.ndarray, ld: int, offset: int, fill: float):
    """Flat device buffer: `offset` floats of fill, rows of `ld` floats (padding = fill),
    then GUARD floats of fill. Returns (buffer, device address of element (0, 0))."""
    rows, cols = host.shape
    flat = torch.full((offset + max(rows, 1) * ld + GUARD,), fill, dtype=torch.float32,
                      device="cuda")
    if rows and cols:
        view = flat[offset:offset + rows * ld].view(rows, ld)
        view[:, :cols] = torch.from_numpy(np.ascontiguousarray(host)).cuda()
    return flat, flat.data_ptr() + 4 * offset


def run(case: Case, entry, torch, check=True, stream=None):
    """Runs `entry` (a binding function with the sgemm signature) on the case and returns
    (normalised error, result rows on host, reference rows)."""
    import dense_fp32_gemm_08_gb300 as sg
    A, B, C = inputs(case)
    M, N, K = case.M, case.N, case.K
    # A and B padding holds NaN: a read past the logical edge poisons the result.
    dA, pA = to_device(torch, A, case.lda, case.a_off, float("nan"))
    dB, pB = to_device(torch, B, case.ldb, case.b_off, float("nan"))
    dC, pC = to_device(torch, C, case.ldc, case.c_off, SENTINEL)
    entry(M, N, K, case.alpha, pA, case.lda, pB, case.ldb, case.beta, pC, case.ldc, stream)
    st = sg.sgemm_device_status(stream)
    assert st == sg.SGEMM_OK, f"device status {st}: {sg.sgemm_last_error()}"
    host = dC.cpu().numpy()
    # Guard bands and padding of C keep the sentinel.
    lead = host[:case.c_off]
    body = host[case.c_off:case.c_off + M * case.ldc].reshape(M, case.ldc) if M else np.zeros((0, case.ldc))
    tail = host[case.c_off + M * case.ldc:]
    assert (lead == SENTINEL).all() and (tail == SENTINEL).all(), "write outside C"
    assert (body[:, N:] == SENTINEL).all(), "write into C's row padding"
    got = body[:, :N]
    rows = case.rows
    got_rows = got if rows is None else got[rows]
    if not check:
        return None, got_rows, None
    Ap = A if case.lda == K else synth.padded(A, case.lda, 0.0)
    Bp = B if case.ldb == N else synth.padded(B, case.ldb, 0.0)
    Cp = C if case.ldc == N else synth.padded(C, case.ldc, 0.0)
    ref = oracle.sgemm(M, N, K, case.alpha, Ap, case.lda, Bp, case.ldb, case.beta,
                       Cp if case.beta != 0.0 else None, case.ldc, rows=rows)
    den = oracle.absdot(M, N, K, Ap, case.lda, Bp, case.ldb, rows=rows)
    c_in = C if rows is None else C[rows]
    err = oracle.normalized_error(got_rows, ref, den, case.alpha, case.beta, c_in)
    return err, got_rows, ref


def sample_rows(M: int, n: int = 48, seed: int = 0, tile: int = 128) -> list:
    """First and last rows, the rows of the last (ragged) row tile, and a seeded sample."""
    rng = np.random.default_rng(seed)
    rows = {0, M - 1}
    rows.update(range(max(0, (M - 1) // tile * tile), M))
    rows.update(int(r) for r in rng.integers(0, M, size=n))
    return sorted(r for r in rows if 0 <= r < M)
