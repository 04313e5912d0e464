"""GPU parity of the FP32 SIMT path through the C ABI, against the CPU oracle.

Acceptance: normalised error max |C_gpu - C_ref| / (sum_k |A_ik||B_kj| + |beta||C_ij|) <= 1e-5
on seeded inputs of every workload shape, and bit-exact results on small-integer inputs
whose sums are exact in fp32."""
from __future__ import annotations

import numpy as np
import pytest

from gemm_case import TOL, Case, run, sample_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sg(sgemm_lib):
    sgemm_lib.sgemm_force_config(-1)
    return sgemm_lib


def _check(case, sg, entry=None):
    err, got, ref = run(case, entry or sg.sgemm, torch)
    assert err <= TOL, f"normalised error {err:.3e} > {TOL} for {case}"
    return got, ref


# ---- the workload configurations ---------------------------------------------------------

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


@pytest.mark.parametrize("n", [128, 256, 512, 1024, 2048, 8192, 16384])
def test_square_sweep(sg, n):
    rows = None if n <= 1024 else sample_rows(n, n=16)
    _check(Case(n, n, n, 1.0, 0.0, "uniform", seed=0, rows=rows), sg)


@pytest.mark.parametrize("K,N", [(4096, 12288), (4096, 14336), (14336, 4096), (4096, 32000)])
def test_llm_shapes(sg, K, N):
    _check(Case(16384, N, K, 1.0, 1.0, "llm", seed=0, rows=sample_rows(16384, n=12)), sg)


# ---- exactness ----------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 517, 1029), (4096, 4096, 4096),
                                   (1, 4096, 4096), (4096, 1, 4096), (129, 255, 16384)])
def test_small_int_bit_exact(sg, M, N, K):
    rows = None if M * N <= 1 << 20 else sample_rows(M, n=16)
    got, ref = _check(Case(M, N, K, 1.0, -2.0, "small_int", seed=5, rows=rows), sg)
    assert np.array_equal(got, ref)


def test_identity_exact(sg):
    n = 300
    A = torch.eye(n, device="cuda")
    B = torch.randn(n, 257, device="cuda")
    C = torch.empty(n, 257, device="cuda")
    sg.sgemm(n, 257, n, 1.0, A, n, B, 257, 0.0, C, 257)
    torch.cuda.synchronize()
    assert torch.equal(C, B)


# ---- alpha / beta semantics and degenerate sizes -------------------------------------------

def test_beta_zero_ignores_nan_in_c(sg):
    _check(Case(300, 260, 70, 1.25, 0.0, "normal", seed=3, nan_c_when_beta0=True), sg)


def test_alpha_zero_and_k_zero(sg):
    n = 97
    C = torch.randn(n, n, device="cuda")
    C0 = C.clone()
    A = torch.full((n, n), float("nan"), device="cuda")
    sg.sgemm(n, n, n, 0.0, A, n, A, n, -0.5, C, n)           # A, B not read
    torch.cuda.synchronize()
    assert torch.equal(C, (-0.5 * C0))
    sg.sgemm(n, n, 0, 1.0, None, 1, None, n, 2.0, C, n)      # K = 0: C = beta * C
    torch.cuda.synchronize()
    assert torch.equal(C, (-1.0 * C0))
    C[0, 0] = float("nan")
    sg.sgemm(n, n, 0, 1.0, None, 1, None, n, 0.0, C, n)      # beta = 0: zeros, C not read
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0


def test_degenerate_noops(sg):
    C = torch.full((4, 4), 7.0, device="cuda")
    sg.sgemm(0, 4, 4, 1.0, None, 4, None, 4, 0.0, C, 4)
    sg.sgemm(4, 0, 4, 1.0, None, 4, None, 1, 0.0, C, 4)
    sg.sgemm_strided_batched(4, 4, 4, 1.0, None, 4, 16, None, 4, 16, 0.0, C, 4, 16, 0)
    torch.cuda.synchronize()
    assert (C == 7.0).all()


# ---- layouts: leading dimensions, misalignment, shape fuzz -----------------------------------

@pytest.mark.parametrize("lda_pad,ldb_pad,ldc_pad,a_off,b_off,c_off", [
    (0, 0, 0, 1, 0, 0), (0, 0, 0, 0, 1, 0), (0, 0, 0, 0, 0, 1), (3, 5, 7, 0, 0, 0),
    (4, 4, 4, 0, 0, 0), (1, 2, 3, 1, 2, 3), (8, 0, 0, 0, 0, 2)])
def test_leading_dims_and_misalignment(sg, lda_pad, ldb_pad, ldc_pad, a_off, b_off, c_off):
    _check(Case(333, 291, 457, 0.7, -1.3, "normal", seed=7, lda_pad=lda_pad, ldb_pad=ldb_pad,
                ldc_pad=ldc_pad, a_off=a_off, b_off=b_off, c_off=c_off), sg)


_FUZZ = [1, 2, 3, 5, 7, 8, 9, 31, 33, 63, 65, 127, 129, 255, 257, 521]


@pytest.mark.parametrize("i", range(24))
def test_shape_fuzz(sg, i):
    rng = np.random.default_rng(1000 + i)
    M, N, K = (int(rng.choice(_FUZZ)) for _ in range(3))
    pads = [int(x) for x in rng.integers(0, 3, size=3)]
    offs = [int(x) for x in rng.integers(0, 2, size=3)]
    _check(Case(M, N, K, 0.7, -1.3, "normal", seed=i, lda_pad=pads[0], ldb_pad=pads[1],
                ldc_pad=pads[2], a_off=offs[0], b_off=offs[1], c_off=offs[2]), sg)


# ---- skinny shapes: one output dimension of at most 8 (bandwidth kernels) ------------------------

@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (2, 1000, 3000), (3, 257, 129), (5, 3001, 77),
                                   (8, 4097, 1025), (4096, 1, 4096), (1000, 2, 3000),
                                   (257, 3, 129), (3001, 7, 77), (4097, 8, 1025), (1, 1, 5000),
                                   (7, 5, 33)])
@pytest.mark.parametrize("pad,off", [(0, 0), (3, 1)])
def test_skinny_shapes(sg, M, N, K, pad, off):
    _check(Case(M, N, K, 0.7, -1.3, "normal", seed=M + N, lda_pad=pad, ldb_pad=pad, ldc_pad=pad,
                a_off=off, b_off=off, c_off=off), sg)
    got, ref = _check(Case(M, N, K, 1.0, 1.0, "small_int", seed=M * N, lda_pad=pad,
                           a_off=off, b_off=off), sg)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("M,N,K,batch", [(1, 640, 300, 4), (500, 3, 200, 3)])
def test_skinny_strided_batched(sg, M, N, K, batch):
    _batched(sg, M, N, K, batch, M * K + 8, K * N + 4, M * N + 4, 0.7, -1.3,
             sg.sgemm_strided_batched)


# ---- every configuration of the table ---------------------------------------------------------

@pytest.mark.parametrize("cfg", range(25))
@pytest.mark.parametrize("shape", [(640, 768, 544), (257, 383, 129), (128, 256, 32),
                                   (4096, 2560, 320), (1000, 3000, 2000)])
def test_each_config(sg, cfg, shape):
    if cfg >= sg.sgemm_num_configs():
        pytest.skip("no such configuration")
    sg.sgemm_force_config(cfg)
    try:
        M, N, K = shape
        _check(Case(M, N, K, 1.5, -0.5, "uniform", seed=cfg), sg)
        got, ref = _check(Case(M, N, K, 1.0, 1.0, "small_int", seed=cfg), sg)
        assert np.array_equal(got, ref)
    finally:
        sg.sgemm_force_config(-1)


@pytest.mark.parametrize("name", ["sk_tma_ws_128x256_s4", "sk_tma_ws_256x128_s4",
                                  "sk_tma_ws_128x128_s3", "sk_cpasync_128x256_s4",
                                  "sk_cpasync_256x128_s4", "packed_sk_tma_128x256_s4",
                                  "sk_tma_ws_128x256_k64_s2", "sk_tma_ws_256x128_k64_s2",
                                  "packed_sk_tma_256x128_k64_s2"])
def test_stream_k_deterministic_and_exact(sg, name):
    ids = {sg.sgemm_config_name(i): i for i in range(sg.sgemm_num_configs())}
    sg.sgemm_force_config(ids[name])
    try:
        # 4096 x 4096: 512 (or 1024) tiles, a data-parallel phase plus a stream-K tail
        case = Case(4096, 4096, 4096, 1.0, 0.0, "uniform", seed=11, rows=sample_rows(4096))
        err, first, ref = run(case, sg.sgemm, torch)
        assert err <= TOL
        _, second, _ = run(case, sg.sgemm, torch, check=False)
        assert np.array_equal(first, second), "stream-K result differs between runs"
        got, ref = _check(Case(2304, 1792, 1000, 1.0, -1.0, "small_int", seed=12,
                               rows=sample_rows(2304)), sg)
        assert np.array_equal(got, ref)
        # unaligned leading dimensions (cp.async loaders take them; TMA ones fall back)
        _check(Case(4095, 3001, 1537, 0.7, -1.3, "normal", seed=13, rows=sample_rows(4095)), sg)
        _check(Case(127, 129, 4099, 0.7, -1.3, "normal", seed=14), sg)
    finally:
        sg.sgemm_force_config(-1)


@pytest.mark.parametrize("name", ["ck_tma_128x256_k64_s2", "ck_tma_256x128_k64_s2",
                                  "packed_ck_tma_128x256_k64_s2", "ck_tma_128x256_s4",
                                  "ck_tma_256x128_s4"])
def test_cluster_k_deterministic_and_exact(sg, name):
    """Cluster split-K: every tile's K slices are added through distributed shared memory in
    rank order, so repeated runs agree bit for bit; small integers are exact. The shapes give
    clusters of 8, 4, 2 and 1 CTAs, fewer k-tiles than slices, ragged edges and a batch."""
    ids = {sg.sgemm_config_name(i): i for i in range(sg.sgemm_num_configs())}
    sg.sgemm_force_config(ids[name])
    try:
        for M, N, K in [(1024, 1024, 1024), (512, 512, 2048), (300, 520, 700), (257, 383, 129),
                        (128, 256, 32), (2048, 2048, 512)]:
            case = Case(M, N, K, 0.7, -1.3, "normal", seed=M + K)
            err, first, _ = run(case, sg.sgemm, torch)
            assert err <= TOL
            _, second, _ = run(case, sg.sgemm, torch, check=False)
            assert np.array_equal(first, second), "cluster split-K result differs between runs"
            got, ref = _check(Case(M, N, K, 1.0, -1.0, "small_int", seed=M + N), sg)
            assert np.array_equal(got, ref)
        _check(Case(333, 291, 457, 0.7, -1.3, "normal", seed=7, lda_pad=4, ldb_pad=8, ldc_pad=3,
                    c_off=3), sg)
        _batched(sg, 256, 320, 200, 3, 256 * 200, 200 * 320, 256 * 320, 0.7, -1.3,
                 sg.sgemm_strided_batched)
    finally:
        sg.sgemm_force_config(-1)


def test_small_splitk_deterministic_and_exact(sg):
    """The one-warp split-K kernel: several K slices per tile, the last to finish adds them in
    slice order, so repeated runs agree bit for bit; small integers are exact."""
    ids = {sg.sgemm_config_name(i): i for i in range(sg.sgemm_num_configs())}
    sg.sgemm_force_config(ids["splitk_cpasync_64x64"])
    try:
        for M, N, K in [(256, 256, 4096), (200, 130, 1000), (64, 64, 32), (1, 70, 3000)]:
            case = Case(M, N, K, 0.7, -1.3, "normal", seed=M + K)
            err, first, _ = run(case, sg.sgemm, torch)
            assert err <= TOL
            _, second, _ = run(case, sg.sgemm, torch, check=False)
            assert np.array_equal(first, second), "split-K result differs between runs"
            got, ref = _check(Case(M, N, K, 1.0, -1.0, "small_int", seed=M + N), sg)
            assert np.array_equal(got, ref)
        # unaligned operands
        _check(Case(333, 291, 457, 0.7, -1.3, "normal", seed=7, lda_pad=1, ldb_pad=2, ldc_pad=3,
                    a_off=1, b_off=2, c_off=3), sg)
        # a launch with more tiles after one with more partial-tile storage (120 tiles in 6
        # slices, then 130 tiles in 5): every tile's count must start at zero
        _check(Case(640, 768, 544, 1.0, 0.0, "uniform", seed=21), sg)
        got, ref = _check(Case(640, 832, 160, 1.0, -1.0, "small_int", seed=22), sg)
        assert np.array_equal(got, ref)
        _check(Case(640, 832, 160, 0.7, -1.3, "normal", seed=23), sg)
    finally:
        sg.sgemm_force_config(-1)


# ---- strided batched ----------------------------------------------------------------------

def _batched(sg, M, N, K, batch, sA, sB, sC, alpha, beta, entry, exact=False):
    import oracle
    import synth
    g = np.random.default_rng(M * 7 + N)
    lda, ldb, ldc = K, N, N
    A = synth.normal(1, max(sA * batch, M * lda), 1).reshape(-1)
    B = synth.normal(1, max(sB * batch, K * ldb), 2).reshape(-1)
    C = synth.normal(1, max(sC * batch, M * ldc), 3).reshape(-1)
    if exact:
        A, B, C = (np.round(x * 2).astype(np.float32) for x in (A, B, C))
    dA, dB, dC = (torch.from_numpy(x.copy()).cuda() for x in (A, B, C))
    entry(M, N, K, alpha, dA, lda, sA, dB, ldb, sB, beta, dC, ldc, sC, batch)
    assert sg.sgemm_device_status() == sg.SGEMM_OK
    out = dC.cpu().numpy()
    for b in range(batch):
        a = np.ascontiguousarray(A[b * sA:b * sA + M * lda])
        bb = np.ascontiguousarray(B[b * sB:b * sB + K * ldb])
        c = np.ascontiguousarray(C[b * sC:b * sC + M * ldc])
        ref = oracle.sgemm(M, N, K, alpha, a, lda, bb, ldb, beta, c, ldc)
        den = oracle.absdot(M, N, K, a, lda, bb, ldb)
        got = out[b * sC:b * sC + M * ldc].reshape(M, ldc)[:, :N]
        err = oracle.normalized_error(got, ref, den, alpha, beta, c.reshape(M, ldc)[:, :N])
        assert err <= TOL, f"batch {b}: {err}"
        if exact:
            assert np.array_equal(got, ref)
    del g


def _config_id(sg, name):
    """Configuration id by name (None: the per-shape table's choice)."""
    if name is None:
        return -1
    ids = {sg.sgemm_config_name(i): i for i in range(sg.sgemm_num_configs())}
    return ids[name]


@pytest.mark.parametrize("M,N,K,batch", [(128, 256, 64, 3), (65, 33, 17, 5), (256, 256, 256, 2),
                                         (512, 768, 300, 7)])
@pytest.mark.parametrize("cfg", [None, "sk_tma_ws_128x256_s4", "pdp_tma_ws_128x256_s4",
                                 "sk_tma_ws_128x128_s3"])
def test_strided_batched(sg, M, N, K, batch, cfg):
    sg.sgemm_force_config(_config_id(sg, cfg))
    try:
        _batched(sg, M, N, K, batch, M * K, K * N, M * N, 0.7, -1.3, sg.sgemm_strided_batched)
        _batched(sg, M, N, K, batch, M * K, K * N, M * N, 1.0, 1.0, sg.sgemm_strided_batched,
                 exact=True)
    finally:
        sg.sgemm_force_config(-1)


@pytest.mark.parametrize("cfg", [None, "packed_sk_tma_128x256_s4", "packed_dp_tma_128x128_s3",
                                 "packed_sk_tma_256x128_k64_s2"])
def test_strided_batched_unaligned(sg, cfg):
    # odd leading dimensions and strides: repacked for TMA (or loaded with cp.async)
    sg.sgemm_force_config(_config_id(sg, cfg))
    try:
        M, N, K, batch = 129, 131, 75, 3
        import oracle
        import synth
        lda, ldb, ldc = K + 1, N + 3, N + 1
        sA, sB, sC = M * lda + 5, K * ldb + 7, M * ldc + 1
        A = synth.normal(1, sA * batch, 21).reshape(-1)
        B = synth.normal(1, sB * batch, 22).reshape(-1)
        C = synth.normal(1, sC * batch, 23).reshape(-1)
        dA, dB, dC = (torch.from_numpy(x.copy()).cuda() for x in (A, B, C))
        sg.sgemm_strided_batched(M, N, K, 0.7, dA, lda, sA, dB, ldb, sB, -1.3, dC, ldc, sC, batch)
        assert sg.sgemm_device_status() == sg.SGEMM_OK
        out = dC.cpu().numpy()
        for b in range(batch):
            a = np.ascontiguousarray(A[b * sA:b * sA + M * lda])
            bb = np.ascontiguousarray(B[b * sB:b * sB + K * ldb])
            c = np.ascontiguousarray(C[b * sC:b * sC + M * ldc])
            ref = oracle.sgemm(M, N, K, 0.7, a, lda, bb, ldb, -1.3, c, ldc)
            den = oracle.absdot(M, N, K, a, lda, bb, ldb)
            got = out[b * sC:b * sC + M * ldc].reshape(M, ldc)[:, :N]
            cin = c.reshape(M, ldc)[:, :N]
            assert oracle.normalized_error(got, ref, den, 0.7, -1.3, cin) <= TOL
    finally:
        sg.sgemm_force_config(-1)


def test_strided_batched_broadcast_and_padding(sg):
    # B shared by every problem (strideB = 0), A and C with gaps between problems.
    M, N, K, batch = 96, 160, 72, 4
    _batched(sg, M, N, K, batch, M * K + 12, 0, M * N + 8, 1.0, 0.5, sg.sgemm_strided_batched)


# ---- C without 16-byte rows and beta != 0: the product staged in an aligned scratch ------------
# (problems of at least 2^22 outputs; the pass that applies alpha, beta, bias and the activation
# reads C with 4-byte loads and must leave every value outside the M x N window untouched)

@pytest.mark.parametrize("name", [None, "dp_tma_128x128_s3", "dp_cpasync_128x256_s4",
                                  "sk_tma_ws_256x128_k64_s2", "sk_tma_ws_128x128_s3",
                                  "ck_tma_128x256_k64_s2", "packed_sk_tma_256x128_k64_s2"])
def test_unaligned_c_beta_staged(sg, name):
    sg.sgemm_force_config(_config_id(sg, name))
    try:
        # odd ldc (A and B stay TMA-readable, so the forced TMA kernels run)
        _check(Case(2049, 2052, 516, 0.7, -1.3, "normal", seed=31, ldc_pad=1,
                    rows=sample_rows(2049, n=12)), sg)
        # C's base 4 bytes past a 16-byte boundary; small integers: bit-exact
        got, ref = _check(Case(2048, 2052, 260, 1.0, -2.0, "small_int", seed=32, c_off=1,
                               rows=sample_rows(2048, n=12)), sg)
        assert np.array_equal(got, ref)
    finally:
        sg.sgemm_force_config(-1)


@pytest.mark.parametrize("M,N,K", [(4095, 3001, 1537), (2051, 2049, 300)])
def test_unaligned_c_beta_staged_exact(sg, M, N, K):
    got, ref = _check(Case(M, N, K, 1.0, 3.0, "small_int", seed=33, rows=sample_rows(M, n=16)),
                      sg)
    assert np.array_equal(got, ref)


def test_unaligned_c_beta_staged_batched(sg):
    # 2 x 1025 x 2049 outputs, ldc = 2049, strideC odd
    M, N, K, batch = 1025, 2049, 64, 2
    _batched(sg, M, N, K, batch, M * K, K * N, M * N + 1, 0.7, -1.3, sg.sgemm_strided_batched)
    _batched(sg, M, N, K, batch, M * K, K * N, M * N + 1, 1.0, 1.0, sg.sgemm_strided_batched,
             exact=True)


# ---- device status ---------------------------------------------------------------------------

def test_device_status_clean(sg):
    assert sg.sgemm_device_status() == sg.SGEMM_OK
