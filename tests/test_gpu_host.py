"""sgemm_host: A, B and C in host memory (pinned or pageable), the product computed in chunks
whose copies overlap the device work, checked against the oracle."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from gemm_case import TOL, sample_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _host(a: np.ndarray, pinned: bool):
    """A host tensor holding a copy of `a` (never sharing its memory)."""
    t = torch.from_numpy(np.array(a, dtype=np.float32, copy=True))
    return t.pin_memory() if pinned else t


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("M,N,K,alpha,beta,pad", [
    (1000, 777, 555, 0.7, -1.3, 0), (100, 300, 200, 1.0, 0.0, 0), (1025, 513, 257, 1.5, 0.5, 3),
    (4096, 4096, 4096, 1.0, 0.0, 0), (300, 200, 100, 0.0, 2.0, 0),
    # eight 512-row chunks (the last in two halves), the first in three K slices (256, 384,
    # 360), beta != 0, padded
    (4096, 4864, 1000, 0.7, -1.3, 5), (2049, 1023, 771, 1.0, 1.0, 1)])
def test_host_buffers(sgemm_lib, pinned, M, N, K, alpha, beta, pad):
    A = synth.normal(M, K, 1)
    B = synth.normal(K, N, 2)
    C = synth.normal(M, N, 3)
    lda, ldb, ldc = K + pad, N + pad, N + pad
    Ap, Bp, Cp = synth.padded(A, lda, 0.0), synth.padded(B, ldb, 0.0), synth.padded(C, ldc, 7.0)
    hA, hB, hC = _host(Ap, pinned), _host(Bp, pinned), _host(Cp, pinned)
    sgemm_lib.sgemm_host(M, N, K, alpha, hA, lda, hB, ldb, beta, hC, ldc)
    got = hC.numpy()
    assert (got[:, N:] == 7.0).all(), "write into C's row padding"
    rows = None if M * N <= 1 << 21 else sample_rows(M, n=16)
    ref = oracle.sgemm(M, N, K, alpha, Ap, lda, Bp, ldb, beta, Cp, ldc, rows=rows)
    den = oracle.absdot(M, N, K, Ap, lda, Bp, ldb, rows=rows)
    g = got[:, :N] if rows is None else got[rows, :N]
    c_in = C if rows is None else C[rows]
    assert oracle.normalized_error(g, ref, den, alpha, beta, c_in) <= TOL


def test_host_buffers_small_int_exact(sgemm_lib):
    M, N, K = 700, 300, 2000
    A, B, C = synth.small_int(M, K, 4), synth.small_int(K, N, 5), synth.small_int(M, N, 6)
    hC = _host(C.copy(), True)
    sgemm_lib.sgemm_host(M, N, K, 1.0, _host(A, True), K, _host(B, True), N, -1.0, hC, N)
    want = (A.astype(np.int64) @ B.astype(np.int64) - C.astype(np.int64)).astype(np.float32)
    assert np.array_equal(hC.numpy(), want)
