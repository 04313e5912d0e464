"""GPU parity of the 3xTF32 tensor-core path (tcgen05) through the C ABI, against the oracle,
held to the same normalised-error bound as the SIMT path (1e-5). Small integers (|v| <= 4)
are exact in TF32 (their small part is zero), so those results must be bit-exact."""
from __future__ import annotations

import numpy as np
import pytest

from gemm_case import TOL, Case, run, sample_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sg(sgemm_lib):
    return sgemm_lib


def _check(case, sg):
    err, got, ref = run(case, sg.sgemm_3xtf32, torch)
    assert err <= TOL, f"normalised error {err:.3e} > {TOL} for {case}"
    return got, ref, err


def test_small_first(sg):
    got, ref, err = _check(Case(128, 128, 32, 1.0, 0.0, "small_int", seed=1), sg)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (1.5, -0.5)])
def test_square_256(sg, alpha, beta):
    _check(Case(256, 256, 256, alpha, beta, "uniform", seed=0), sg)


def test_headline_4096(sg):
    _check(Case(4096, 4096, 4096, 1.0, 0.0, "uniform", seed=0, rows=sample_rows(4096)), sg)


@pytest.mark.parametrize("M,N,K", [(4095, 3001, 1537), (1, 4096, 4096), (4096, 1, 4096),
                                   (127, 129, 4099)])
def test_edge_shapes(sg, M, N, K):
    rows = None if M * N <= 4096 * 4096 // 2 else sample_rows(M)
    _check(Case(M, N, K, 0.7, -1.3, "normal", seed=0, rows=rows), sg)


@pytest.mark.parametrize("n", [128, 512, 2048, 8192])
def test_square_sweep(sg, n):
    rows = None if n <= 512 else sample_rows(n, n=16)
    _check(Case(n, n, n, 1.0, 0.0, "uniform", seed=0, rows=rows), sg)


def test_long_k_accuracy(sg):
    # The tensor core accumulates in fp32 inside TMEM; at K = 16384 the error must still be
    # within the bound (measured, not assumed).
    _, _, err = _check(Case(256, 384, 16384, 1.0, 0.0, "normal", seed=4), sg)
    print(f"3xTF32 normalised error at K=16384: {err:.3e}")


@pytest.mark.parametrize("K,N", [(4096, 12288), (14336, 4096)])
def test_llm_shapes(sg, K, N):
    _check(Case(16384, N, K, 1.0, 1.0, "llm", seed=0, rows=sample_rows(16384, n=8)), sg)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 517, 1029), (129, 255, 16384)])
def test_small_int_bit_exact(sg, M, N, K):
    got, ref, _ = _check(Case(M, N, K, 1.0, -2.0, "small_int", seed=5), sg)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("lda_pad,ldb_pad,ldc_pad,a_off,b_off,c_off", [
    (0, 0, 0, 1, 0, 0), (0, 0, 0, 0, 1, 0), (0, 0, 0, 0, 0, 1), (3, 5, 7, 0, 0, 0),
    (1, 2, 3, 1, 2, 3)])
def test_leading_dims_and_misalignment(sg, lda_pad, ldb_pad, ldc_pad, a_off, b_off, c_off):
    _check(Case(333, 291, 457, 0.7, -1.3, "normal", seed=7, lda_pad=lda_pad, ldb_pad=ldb_pad,
                ldc_pad=ldc_pad, a_off=a_off, b_off=b_off, c_off=c_off), sg)


_FUZZ = [1, 2, 3, 5, 7, 8, 9, 31, 33, 63, 65, 127, 129, 255, 257, 521]


@pytest.mark.parametrize("i", range(12))
def test_shape_fuzz(sg, i):
    rng = np.random.default_rng(2000 + i)
    M, N, K = (int(rng.choice(_FUZZ)) for _ in range(3))
    _check(Case(M, N, K, 0.7, -1.3, "normal", seed=i), sg)


def test_beta_zero_ignores_nan_in_c(sg):
    _check(Case(300, 260, 70, 1.25, 0.0, "normal", seed=3, nan_c_when_beta0=True), sg)


def test_strided_batched(sg):
    import oracle
    import synth
    M, N, K, batch = 200, 160, 96, 3
    sA, sB, sC = M * K + 4, K * N, M * N + 8
    A = synth.normal(1, sA * batch, 1).reshape(-1)
    B = synth.normal(1, sB * batch, 2).reshape(-1)
    C = synth.normal(1, sC * batch, 3).reshape(-1)
    dA, dB, dC = (torch.from_numpy(x.copy()).cuda() for x in (A, B, C))
    sg.sgemm_3xtf32_strided_batched(M, N, K, 0.7, dA, K, sA, dB, N, sB, -1.3, dC, N, sC, batch)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    out = dC.cpu().numpy()
    for b in range(batch):
        a = np.ascontiguousarray(A[b * sA:b * sA + M * K])
        bb = np.ascontiguousarray(B[b * sB:b * sB + K * N])
        c = np.ascontiguousarray(C[b * sC:b * sC + M * N])
        ref = oracle.sgemm(M, N, K, 0.7, a, K, bb, N, -1.3, c, N)
        den = oracle.absdot(M, N, K, a, K, bb, N)
        got = out[b * sC:b * sC + M * N].reshape(M, N)
        assert oracle.normalized_error(got, ref, den, 0.7, -1.3, c.reshape(M, N)) <= TOL


@pytest.mark.parametrize("entry,bound", [("sgemm_3xtf32", TOL), ("sgemm_tf32", 1e-3)])
def test_values_near_flt_max_stay_finite(sg, entry, bound):
    # FLT_MAX rounds to Inf under round-to-nearest-away to TF32; the split must keep such a
    # value finite, so the product matches fp32 arithmetic (and the oracle) instead of
    # overflowing. A's first row holds +-FLT_MAX in two places, B's matching rows hold 1/8,
    # so the result stays far from the fp32 limit.
    import oracle
    import synth
    M, N, K = 64, 96, 80
    fmax = float(np.finfo(np.float32).max)
    A = synth.normal(M, K, 70)
    B = synth.normal(K, N, 71)
    A[0, 3], A[5, 40] = fmax, -fmax
    B[3, :] = 0.125
    B[40, :] = 0.125
    C = np.zeros((M, N), np.float32)
    dA, dB, dC = (torch.from_numpy(x.copy()).cuda() for x in (A, B, C))
    getattr(sg, entry)(M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    got = dC.cpu().numpy()
    assert np.isfinite(got).all(), f"{entry}: non-finite result from finite inputs"
    ref = oracle.sgemm(M, N, K, 1.0, A, K, B, N, 0.0, None, N)
    den = oracle.absdot(M, N, K, A, K, B, N)
    assert oracle.normalized_error(got, ref, den, 1.0, 0.0, None) <= bound
