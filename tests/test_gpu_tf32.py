"""GPU parity of the single-product TF32 mode (sgemm_tf32) through the C ABI.

Tolerance, derived from the arithmetic: each operand is rounded to TF32 (round to nearest,
unit roundoff u = 2^-11), so each product a*b is replaced by a(1+d1)*b(1+d2) with |d| <= u,
an error of at most (2u + u^2)|a b| = 9.77e-4 |a b|. Summed over k and divided by
sum_k |a||b|, that is at most 9.77e-4, plus the fp32 accumulation (measured below 2e-6 at
K = 16384 on the 3xTF32 path that shares the kernel). The bound checked is 1e-3. Small
integers are exact in TF32, so those results must be bit-exact."""
from __future__ import annotations

import numpy as np
import pytest

from gemm_case import Case, run, sample_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TOL_TF32 = 1e-3


def _check(case, sg):
    err, got, ref = run(case, sg.sgemm_tf32, torch)
    assert err <= TOL_TF32, f"normalised error {err:.3e} > {TOL_TF32} for {case}"
    return got, ref, err


def test_small_first(sgemm_lib):
    got, ref, _ = _check(Case(128, 128, 32, 1.0, 0.0, "small_int", seed=1), sgemm_lib)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (1.5, -0.5)])
def test_square_256(sgemm_lib, alpha, beta):
    _check(Case(256, 256, 256, alpha, beta, "uniform", seed=0), sgemm_lib)


def test_headline_4096(sgemm_lib):
    _, _, err = _check(Case(4096, 4096, 4096, 1.0, 0.0, "uniform", seed=0,
                            rows=sample_rows(4096)), sgemm_lib)
    print(f"1xTF32 normalised error at 4096^3: {err:.3e}")


@pytest.mark.parametrize("M,N,K", [(4095, 3001, 1537), (1, 4096, 4096), (4096, 1, 4096),
                                   (127, 129, 4099), (256, 384, 16384)])
def test_edge_and_long_k(sgemm_lib, M, N, K):
    rows = None if M * N <= 4096 * 4096 // 2 else sample_rows(M)
    _check(Case(M, N, K, 0.7, -1.3, "normal", seed=0, rows=rows), sgemm_lib)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 517, 1029), (129, 255, 16384)])
def test_small_int_bit_exact(sgemm_lib, M, N, K):
    got, ref, _ = _check(Case(M, N, K, 1.0, -2.0, "small_int", seed=5), sgemm_lib)
    assert np.array_equal(got, ref)


def test_misaligned(sgemm_lib):
    _check(Case(333, 291, 457, 0.7, -1.3, "normal", seed=7, lda_pad=1, ldb_pad=2, ldc_pad=3,
                a_off=1, b_off=2, c_off=3), sgemm_lib)


def test_strided_batched(sgemm_lib):
    import oracle
    import synth
    sg = sgemm_lib
    M, N, K, batch = 200, 160, 96, 3
    sA, sB, sC = M * K + 4, K * N, M * N + 8
    A = synth.normal(1, sA * batch, 1).reshape(-1)
    B = synth.normal(1, sB * batch, 2).reshape(-1)
    C = synth.normal(1, sC * batch, 3).reshape(-1)
    dA, dB, dC = (torch.from_numpy(x.copy()).cuda() for x in (A, B, C))
    sg.sgemm_tf32_strided_batched(M, N, K, 0.7, dA, K, sA, dB, N, sB, -1.3, dC, N, sC, batch)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    out = dC.cpu().numpy()
    for b in range(batch):
        a = np.ascontiguousarray(A[b * sA:b * sA + M * K])
        bb = np.ascontiguousarray(B[b * sB:b * sB + K * N])
        c = np.ascontiguousarray(C[b * sC:b * sC + M * N])
        ref = oracle.sgemm(M, N, K, 0.7, a, K, bb, N, -1.3, c, N)
        den = oracle.absdot(M, N, K, a, K, bb, N)
        got = out[b * sC:b * sC + M * N].reshape(M, N)
        assert oracle.normalized_error(got, ref, den, 0.7, -1.3, c.reshape(M, N)) <= TOL_TF32


# The persistent kernel picks its tile width (192, 224 or 256 columns) from the number of
# rounds of tiles the grid needs; each shape below selects one width and gives every CTA
# at least three tiles, so both TMEM accumulator sets are reused.
@pytest.mark.parametrize("M,N,width", [(1280, 7744, 192), (1408, 7936, 224), (1664, 7872, 256)])
def test_each_tile_width(sgemm_lib, M, N, width):
    got, ref, _ = _check(Case(M, N, 64, 1.0, -1.0, "small_int", seed=11), sgemm_lib)
    assert np.array_equal(got, ref)
    _check(Case(M, N, 200, 0.7, 0.5, "normal", seed=12, rows=sample_rows(M)), sgemm_lib)
