"""sgemm_noalloc: the entry point for callers that must not have the library allocate device
memory (their memory budget belongs to their own pool, or they cannot take the
synchronisation that cudaMalloc / cudaFree may cause). Its scratch is a static array in the
library. Through the C ABI, two calls in a row must each agree with the oracle (on a sample
of rows) and with sgemm() (on the whole matrix) on the same inputs, within the
normalised-error bound every GPU test here uses, and must leave the device's free memory
unchanged.

This file is collected last on purpose: if it fails, every other test has already run."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

from gemm_case import TOL

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("M,N,K,alpha,beta", [
    (4096, 4096, 4096, 1.0, 0.0),    # data-parallel waves plus a stream-K tail
    (2048, 3072, 1000, 0.7, -1.3),   # stream-K over every tile
    (300, 520, 700, 1.5, 0.5),       # fewer tiles than SMs, ragged edges
])
def test_noalloc_matches_sgemm_twice(sgemm_lib, M, N, K, alpha, beta):
    import oracle
    import synth
    L = sgemm_lib.lib()
    A = synth.uniform(M, K, 40)
    B = synth.uniform(K, N, 41)
    C = synth.uniform(M, N, 42)
    dA, dB = _to_dev(A), _to_dev(B)
    stream = torch.cuda.current_stream().cuda_stream

    ref = _to_dev(C)
    st = L.sgemm(M, N, K, ctypes.c_float(alpha), dA.data_ptr(), K, dB.data_ptr(), N,
                 ctypes.c_float(beta), ref.data_ptr(), N, stream)
    assert st == 0, L.sgemm_last_error()
    assert L.sgemm_device_status(stream) == 0
    ref_h = ref.cpu().numpy()

    # The oracle on a sample of rows: first, last, the last row tile and an even spread.
    rows = np.unique(np.r_[0, M - 1, np.arange(max(0, M - 128), M, 37),
                          np.linspace(0, M - 1, 24).astype(int)])
    want = oracle.sgemm(M, N, K, alpha, A, K, B, N, beta, C, N, rows=rows)
    den = oracle.absdot(M, N, K, A, K, B, N, rows=rows)

    # Every buffer exists before the calls under test; one warm-up call does the per-device
    # set-up (the array's address, kernel attributes, the module's first load).
    outs = [_to_dev(C) for _ in range(3)]
    st = L.sgemm_noalloc(M, N, K, ctypes.c_float(alpha), dA.data_ptr(), K, dB.data_ptr(), N,
                         ctypes.c_float(beta), outs[2].data_ptr(), N, stream)
    assert st == 0, f"warm-up call: {L.sgemm_last_error()}"
    assert L.sgemm_device_status(stream) == 0
    free_before = torch.cuda.mem_get_info()[0]
    for call in range(2):
        st = L.sgemm_noalloc(M, N, K, ctypes.c_float(alpha), dA.data_ptr(), K, dB.data_ptr(), N,
                             ctypes.c_float(beta), outs[call].data_ptr(), N, stream)
        assert st == 0, f"call {call}: {L.sgemm_last_error()}"
        assert L.sgemm_device_status(stream) == 0, f"call {call}: device status"
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before, "device memory changed across the no-allocation calls"

    for call in range(2):
        got = outs[call].cpu().numpy()
        assert np.isfinite(got).all()
        # against the oracle, within the bound every GPU test here uses
        err = oracle.normalized_error(got[rows], want, den, alpha, beta, C[rows])
        assert err <= TOL, f"call {call}: normalised error {err:.3e} against the oracle"
        # and against sgemm(), the entry point it stands in for, on the whole matrix
        scale = np.abs(A).sum(axis=1, keepdims=True) * np.abs(B).max() + abs(beta) * np.abs(C)
        assert (np.abs(got - ref_h) <= TOL * scale).all(), f"call {call}: differs from sgemm()"


def test_noalloc_rejects_unaligned_operands(sgemm_lib):
    L = sgemm_lib.lib()
    M = N = K = 64
    buf = torch.zeros(M * K + 1, device="cuda")
    C = torch.zeros(M, N, device="cuda")
    st = L.sgemm_noalloc(M, N, K, ctypes.c_float(1.0), buf.data_ptr() + 4, K, buf.data_ptr(), N,
                         ctypes.c_float(0.0), C.data_ptr(), N, None)
    assert st == 4  # SGEMM_ERR_UNSUPPORTED
    assert "aligned" in L.sgemm_last_error().decode()
