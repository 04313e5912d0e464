"""GPU parity of the fused epilogue, C = act(alpha * op(A) op(B) + bias) + beta * C, through
sgemm_fused on every path and configuration, against the oracle's plainly written epilogue.

Tolerance. Let x = alpha * op(A) op(B) + bias be the pre-activation value; its fp32 error is
that of the plain product, bounded by the path's bound times |alpha| sum_k |a||b| + |bias|
(the bias add rounds once more, a fraction of an ulp of |x|). The activation passes that
error on scaled by its Lipschitz constant (1 for identity and ReLU, at most 1.13 for the two
GELU forms, 1.1 for SiLU) and adds the error of its own fp32 evaluation: a few ulps of the
larger of |x| and 1 times |x| at worst (CUDA documents erff, tanhf and expf to within 2 ulps;
the surrounding multiply-adds add about one ulp each), about 8 * 2^-24 |x| = 4.8e-7 |x|. So
each cell is judged against
    L * (|alpha| sum_k |a||b| + |bias|) + |beta| |C|
with L = 1 for act = none (the plain product's bound with the bias in the denominator) and
L = 1.2 for the activations (1.13 for the input error plus 0.07 * bound >= 4.8e-7 for the
activation's own rounding at the 1e-5 bound), and the ratio must stay below the path's bound
(1e-5 for the SIMT and 3xTF32 paths, 1e-3 for the TF32 path)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from gemm_case import TOL

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ACTS = ["none", "relu", "gelu", "gelu_tanh", "silu"]
PATH_TOL = {"simt": TOL, "3xtf32": TOL, "tf32": 1e-3}
LIPSCHITZ = 1.2


def fused_error(got, ref, den, alpha, beta, c_in, bias, act):
    b = 0.0 if bias is None else np.abs(bias.astype(np.float64))[None, :]
    lip = 1.0 if act == "none" else LIPSCHITZ
    scale = lip * (abs(alpha) * den + b) + abs(beta) * np.abs(c_in.astype(np.float64))
    diff = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    both_nan = np.isnan(got) & np.isnan(ref)
    diff = np.where(both_nan, 0.0, diff)
    if np.isnan(diff).any():
        return float("inf")
    zero = scale == 0
    if (diff[zero] != 0).any():
        return float("inf")
    return float((diff[~zero] / scale[~zero]).max()) if (~zero).any() else 0.0


def _run(sg, M, N, K, alpha, beta, act, with_bias, path="simt", ta=False, tb=False, seed=0,
         dist="normal", rows=None):
    gen = synth.small_int if dist == "small_int" else synth.normal
    A = gen(M, K, seed)
    B = gen(K, N, seed + 1)
    C = gen(M, N, seed + 2)
    bias = gen(1, N, seed + 3).reshape(-1) if with_bias else None
    As = np.ascontiguousarray(A.T) if ta else A
    Bs = np.ascontiguousarray(B.T) if tb else B
    lda, ldb = max(As.shape[1], 1), max(Bs.shape[1], 1)
    As = As if As.size else np.zeros((As.shape[0], 1), np.float32)
    Bs = Bs if Bs.size else np.zeros((max(Bs.shape[0], 1), 1), np.float32)
    dA, dB, dC = (torch.from_numpy(x.copy()).cuda() for x in (As, Bs, C))
    dbias = None if bias is None else torch.from_numpy(bias.copy()).cuda()
    sg.sgemm_fused("T" if ta else "N", "T" if tb else "N", M, N, K, alpha, dA, lda, dB, ldb, beta,
                   dC, N, bias=dbias, act=act, path=path)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    got = dC.cpu().numpy()
    idx = slice(None) if rows is None else rows
    ref = oracle.sgemm_epilogue(ta, tb, M, N, K, alpha, As, lda, Bs, ldb, beta, C, N, bias, act,
                                rows=rows)
    den = oracle.absdot_ex(ta, tb, M, N, K, As, lda, Bs, ldb, rows=rows)
    err = fused_error(got[idx], ref, den, alpha, beta, C[idx], bias, act)
    assert err <= PATH_TOL[path], f"{path} act={act} bias={with_bias}: {err:.3e}"
    return got[idx], ref


@pytest.mark.parametrize("path", ["simt", "3xtf32", "tf32"])
@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.7, 1.0)])
def test_fused_epilogue(sgemm_lib, path, act, with_bias, alpha, beta):
    _run(sgemm_lib, 384, 640, 512, alpha, beta, act, with_bias, path=path, seed=7)


@pytest.mark.parametrize("cfg", range(25))
def test_fused_every_config(sgemm_lib, cfg):
    sg = sgemm_lib
    if cfg >= sg.sgemm_num_configs():
        pytest.skip("no such configuration")
    name = sg.sgemm_config_name(cfg)
    shape = (4096, 3, 300) if "tall" in name else (3, 2000, 300) if "wide" in name else (1000, 3000, 700)
    sg.sgemm_force_config(cfg)
    try:
        _run(sg, *shape, 1.0, 1.0, "gelu", True, seed=cfg)
        got, ref = _run(sg, *shape, 1.0, 1.0, "relu", True, seed=cfg, dist="small_int")
        assert np.array_equal(got, ref)
    finally:
        sg.sgemm_force_config(-1)


@pytest.mark.parametrize("ta,tb", [(True, False), (False, True), (True, True)])
def test_fused_transposed(sgemm_lib, ta, tb):
    _run(sgemm_lib, 300, 500, 257, 0.7, 1.0, "silu", True, ta=ta, tb=tb, seed=11)


def test_fused_alpha_zero_is_act_of_bias(sgemm_lib):
    _run(sgemm_lib, 64, 96, 32, 0.0, 0.5, "gelu", True, seed=13)
    _run(sgemm_lib, 64, 96, 0, 1.0, 0.0, "silu", True, seed=14)


def test_fused_llm_ffn_up_gelu(sgemm_lib):
    rows = sorted({0, 16383, *range(16256, 16384, 37), *np.random.default_rng(0).integers(0, 16384, 8).tolist()})
    _run(sgemm_lib, 16384, 14336, 4096, 1.0, 0.0, "gelu", True, seed=0, rows=rows)


@pytest.mark.parametrize("act", ["relu", "gelu", "silu"])
def test_fused_unaligned_c_staged(sgemm_lib, act):
    # ldc = 2049 (odd) and beta != 0 over 4.2 M outputs: the product is staged in an aligned
    # scratch and the bias, activation and beta * C are applied by a separate pass
    rows = sorted({0, 2048, *range(1920, 2049, 41), *np.random.default_rng(1).integers(0, 2049, 8).tolist()})
    _run(sgemm_lib, 2049, 2049, 300, 0.7, -1.3, act, True, seed=4, rows=rows)
    got, ref = _run(sgemm_lib, 2049, 2049, 300, 1.0, 2.0, "relu" if act == "relu" else "none",
                    True, seed=5, dist="small_int", rows=rows)
    assert np.array_equal(got, ref)


def test_fused_strided_batched(sgemm_lib):
    sg = sgemm_lib
    M, N, K, batch = 200, 160, 96, 3
    A = synth.normal(1, M * K * batch, 1).reshape(-1)
    B = synth.normal(1, K * N * batch, 2).reshape(-1)
    C = synth.normal(1, M * N * batch, 3).reshape(-1)
    bias = synth.normal(1, N, 4).reshape(-1)
    dA, dB, dC, db = (torch.from_numpy(x.copy()).cuda() for x in (A, B, C, bias))
    sg.sgemm_fused_strided_batched("N", "N", M, N, K, 0.7, dA, K, M * K, dB, N, K * N, 1.0, dC, N,
                                   M * N, batch, bias=db, act="gelu_tanh")
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    out = dC.cpu().numpy().reshape(batch, M, N)
    for b in range(batch):
        a = np.ascontiguousarray(A[b * M * K:(b + 1) * M * K]).reshape(M, K)
        bb = np.ascontiguousarray(B[b * K * N:(b + 1) * K * N]).reshape(K, N)
        c = np.ascontiguousarray(C[b * M * N:(b + 1) * M * N]).reshape(M, N)
        ref = oracle.sgemm_epilogue(False, False, M, N, K, 0.7, a, K, bb, N, 1.0, c, N, bias,
                                    "gelu_tanh")
        den = oracle.absdot(M, N, K, a, K, bb, N)
        assert fused_error(out[b], ref, den, 0.7, 1.0, c, bias, "gelu_tanh") <= TOL
