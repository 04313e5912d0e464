"""GPU parity of sgemm_ex / sgemm_ex_strided_batched: transposed operands (op(A) = A^T with A
stored K x M, op(B) = B^T with B stored N x K) on each arithmetic path, against the oracle's
transposed entry. Same bounds as the plain entry points: 1e-5 for the SIMT and 3xTF32 paths,
the derived 1e-3 for the single-product TF32 path; small integers bit-exact everywhere."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from gemm_case import TOL

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PATH_TOL = {"simt": TOL, "3xtf32": TOL, "tf32": 1e-3}


def _stored(mat: np.ndarray, trans: bool, pad: int) -> tuple[np.ndarray, int]:
    """Storage of op(X) = mat: mat itself, or its transpose, with `pad` extra columns."""
    s = np.ascontiguousarray(mat.T) if trans else mat
    ld = s.shape[1] + pad
    return synth.padded(s, ld, np.nan), ld


def _run(sg, path, ta, tb, M, N, K, alpha, beta, dist="normal", pad=0, off=0, seed=0):
    gen = synth.small_int if dist == "small_int" else synth.normal
    A = gen(M, K, seed)          # op(A), M x K
    B = gen(K, N, seed + 1)      # op(B), K x N
    C = gen(M, N, seed + 2)
    As, lda = _stored(A, ta, pad)
    Bs, ldb = _stored(B, tb, pad)
    dA = torch.full((As.size + off + 16,), float("nan"), device="cuda")
    dB = torch.full((Bs.size + off + 16,), float("nan"), device="cuda")
    dA[off:off + As.size] = torch.from_numpy(As.reshape(-1)).cuda()
    dB[off:off + Bs.size] = torch.from_numpy(Bs.reshape(-1)).cuda()
    dC = torch.from_numpy(C.copy()).cuda()
    sg.sgemm_ex("T" if ta else "N", "T" if tb else "N", M, N, K, alpha, dA.data_ptr() + 4 * off,
                lda, dB.data_ptr() + 4 * off, ldb, beta, dC, N, path=path)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    got = dC.cpu().numpy()
    As0 = np.where(np.isnan(As), 0.0, As).astype(np.float32)
    Bs0 = np.where(np.isnan(Bs), 0.0, Bs).astype(np.float32)
    ref = oracle.sgemm_ex(ta, tb, M, N, K, alpha, As0, lda, Bs0, ldb, beta, C, N)
    den = oracle.absdot_ex(ta, tb, M, N, K, As0, lda, Bs0, ldb)
    err = oracle.normalized_error(got, ref, den, alpha, beta, C)
    assert err <= PATH_TOL[path], f"{path} ta={ta} tb={tb}: {err:.3e}"
    return got, ref


@pytest.mark.parametrize("path", ["simt", "3xtf32", "tf32"])
@pytest.mark.parametrize("ta,tb", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K,pad,off", [(256, 384, 320, 0, 0), (333, 291, 457, 3, 1),
                                           (1, 500, 300, 0, 0), (500, 3, 300, 1, 0)])
def test_transposed_operands(sgemm_lib, path, ta, tb, M, N, K, pad, off):
    _run(sgemm_lib, path, ta, tb, M, N, K, 0.7, -1.3, pad=pad, off=off, seed=M + N)


@pytest.mark.parametrize("path", ["simt", "3xtf32", "tf32"])
@pytest.mark.parametrize("ta,tb", [(True, False), (False, True), (True, True)])
def test_transposed_small_int_exact(sgemm_lib, path, ta, tb):
    got, ref = _run(sgemm_lib, path, ta, tb, 640, 384, 1000, 1.0, 1.0, dist="small_int", seed=3)
    assert np.array_equal(got, ref)


def test_transposed_large(sgemm_lib):
    _run(sgemm_lib, "simt", True, True, 2048, 2048, 2048, 1.0, 0.0, seed=5)


@pytest.mark.parametrize("ta,tb", [(True, False), (False, True)])
def test_transposed_unaligned_c_staged(sgemm_lib, ta, tb):
    # ldc = N = 2051 (odd), beta != 0 and 4.2 M outputs: the untransposed product is staged in
    # an aligned scratch and a second pass applies alpha and beta to C
    _run(sgemm_lib, "simt", ta, tb, 2049, 2051, 300, 0.7, -1.3, seed=7)
    got, ref = _run(sgemm_lib, "simt", ta, tb, 2049, 2051, 300, 1.0, 2.0, dist="small_int",
                    seed=8)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("path", ["simt", "3xtf32"])
def test_transposed_strided_batched(sgemm_lib, path):
    sg = sgemm_lib
    M, N, K, batch = 96, 80, 72, 3
    A = [synth.normal(M, K, 30 + b) for b in range(batch)]
    B = [synth.normal(K, N, 40 + b) for b in range(batch)]
    C = [synth.normal(M, N, 50 + b) for b in range(batch)]
    At = np.concatenate([np.ascontiguousarray(a.T).reshape(-1) for a in A])   # K x M each
    Bt = np.concatenate([np.ascontiguousarray(b.T).reshape(-1) for b in B])   # N x K each
    Cc = np.concatenate([c.reshape(-1) for c in C])
    dA, dB, dC = (torch.from_numpy(x.copy()).cuda() for x in (At, Bt, Cc))
    sg.sgemm_ex_strided_batched("T", "T", M, N, K, 0.7, dA, M, K * M, dB, K, N * K, -1.3, dC, N,
                                M * N, batch, path=path)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    out = dC.cpu().numpy().reshape(batch, M, N)
    for b in range(batch):
        ref = oracle.sgemm(M, N, K, 0.7, A[b], K, B[b], N, -1.3, C[b], N)
        den = oracle.absdot(M, N, K, A[b], K, B[b], N)
        assert oracle.normalized_error(out[b], ref, den, 0.7, -1.3, C[b]) <= TOL
