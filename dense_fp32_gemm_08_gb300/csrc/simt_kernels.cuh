// simt_kernels.cuh: the FP32 SIMT kernels of sm_103a as templates, with their launch
// templates, for the translation units that instantiate them (simt_gemm_*.cu; one unit per group
// of configurations, so the large unrolled kernels compile in parallel) and for simt_gemm.cu,
// which holds the host-side state they share (workspaces, device queries, tensor maps), the
// configuration table and the small kernels. C = alpha * (A . B) + beta * C, row-major.
//
//
// Design (the tiling ladder of the "GEMM scrapbook" re-done for GB300):
//  * CTA tile BM x BN, k-tile BK = 32, staged in a STAGES-deep shared-memory ring
//    ("double buffering", generalised). The A and B k-tiles arrive by TMA
//    (cp.async.bulk.tensor, completion on an mbarrier) when both operands are 16-byte
//    aligned with leading dimensions that are multiples of 4, otherwise by cp.async with
//    zero fill. TMA's out-of-bounds fill and cp.async's zero fill supply the zeros of
//    ragged M, N and K edges, so the compute loop never branches on edges.
//  * Warp tile 64 x 64 ("warptiling" chapter), thread tile 8 x 16 (the "2D block-tiling"
//    outer product: per k, a sliver of 8 A values and 16 B values gives 128 multiply-adds).
//    The multiply-adds are issued as paired fp32 FMAs (__ffma2_rn, two independent FMAs per
//    instruction), which halves the issue slots the FMA stream needs on Blackwell and leaves
//    room for the shared-memory loads. Each output cell still accumulates in fp32 with one
//    rounding per FMA, in ascending k.
//  * Shared-memory layout without bank conflicts ("bank-conflict dodging"):
//    - A tile: BM rows of 32 floats (128 B), the 16-byte chunk c of row m stored at chunk
//      c ^ (m & 7) (the 128-byte TMA swizzle; the cp.async loader writes the same layout).
//      Thread row tr owns rows tr, tr + 8, ..., tr + 56 of its warp tile, so the 8 rows one
//      LDS.128 touches sit in 8 different chunk columns.
//    - B tile: 32 rows of BN floats, unswizzled; the 4 column threads of a warp read 4
//      adjacent 16-byte chunks (cols 16q + 4tc).
//    - A values are read as float4 along k (4 k-steps per load), B values as float4 along n
//      ("float4" chapter: 128-bit loads), no transposed copy of A is needed.
//  * Epilogue: alpha * acc + beta * C fused, float4 loads and stores where C allows,
//    C never read when beta == 0.
//  * Schedules: a data-parallel grid (one CTA per tile); a persistent grid (one CTA per SM,
//    or two) that deals whole tiles round-robin and splits the last partial wave's tiles
//    along K (stream-K, deterministic fixed-order fix-up); persistent variants whose stages
//    hold two 32-wide k-tiles (one CTA barrier per 64 k-steps); and, for outputs of at most
//    512 x 512, one warp per 64 x 64 tile with K split over CTAs. Which one runs is decided
//    per shape class by measured sweeps (config_table.h).
#pragma once

#include "epilogue.cuh"
#include "ptx.cuh"
#include "raster.cuh"
#include "simt_gemm.cuh"

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

namespace sg {

// ---- host-side helpers shared by the kernel units (defined in simt_gemm.cu) -----------------

constexpr int kMaxDevices = 64;
constexpr size_t kFlagBytes = 64 * 1024;  // stream-K flags: room for 2048 CTAs x 8 warps

// rows x cols fp32 matrix with leading dimension ld, `batch` copies `stride` elements apart,
// read in boxes of box_rows x box_cols (optionally with the 128-byte swizzle).
bool make_map(CUtensorMap *map, const float *base, long long rows, long long cols, long long ld,
              long long stride, int batch, int box_rows, int box_cols, bool swizzle128);
// 16-byte aligned base, leading dimension and batch stride multiples of 4 elements.
bool operand_vec4(const float *ptr, long long ld, long long stride, int batch);
// Both operands readable by TMA in place.
bool tma_ok(const SimtProblem &p);
// Multiprocessors of device `dev` (cached), 0 when the query fails.
int device_sms(int dev);
// The stream-K workspace of (dev, stream): kFlagBytes of flags, then `partial_bytes` of partial
// sums; returns the next flag epoch of that workspace through `epoch`.
cudaError_t workspace_for(int dev, cudaStream_t stream, size_t partial_bytes, float4 **ws,
                          unsigned int **flags, unsigned int *epoch);
// k-tiles per CTA when a stream-K grid of under one wave splits every tile along K.
int sk_min_iters_per_cta(long long KT, int KSUB);
// CTAs per cluster of the cluster split-K schedule.
int clusterk_slices(long long tiles, int KT, int sms);

// ---- launchers of the kernel units (configuration ids as in simt_gemm.cu's table) ----------

cudaError_t simt_launch_dp(int id, const SimtProblem &p, cudaStream_t stream, const char **detail);
cudaError_t simt_launch_dpcp(int id, const SimtProblem &p, cudaStream_t stream,
                             const char **detail);
cudaError_t simt_launch_sk(int id, const SimtProblem &p, cudaStream_t stream, const char **detail);
cudaError_t simt_launch_sk128(int id, const SimtProblem &p, cudaStream_t stream,
                              const char **detail);
cudaError_t simt_launch_sk64(int id, const SimtProblem &p, cudaStream_t stream,
                             const char **detail);
cudaError_t simt_launch_skcp(int id, const SimtProblem &p, cudaStream_t stream,
                             const char **detail);
cudaError_t simt_launch_ck(int id, const SimtProblem &p, cudaStream_t stream, const char **detail);

namespace {

constexpr int BK = 32;

struct KParams {
    int M, N, K;
    float alpha, beta;
    const float *A;
    const float *B;
    float *C;
    long long lda, ldb, ldc;
    long long sA, sB, sC;
    int batch;
    int tiles_m, tiles_n, group_m;
    int a_vec4, b_vec4, c_vec4;
    const float *bias;  // fused epilogue (nullptr: none)
    int act;            // fused epilogue activation (0: none)
};

// Orders in which one k-step's 64 paired FMAs of a thread tile are issued. Every accumulator
// still sums its k-steps in ascending order, so all orders give identical results; they
// differ in how ptxas interleaves the FMAs with the next fragment loads. Measured on a GB300
// at 4096^3 (TFLOP/s, row-outer order / these orders): data-parallel 128x128 62.3 / 63.8 with
// kOrderHalfSnake, stream-K 128x256 with 32-wide stages 62.4 / 63.0 with kOrderHalfSnake,
// stream-K 128x256 with 64-wide stages 63.9 / 65.2 with kOrderColumnSnake (64.7 with
// kOrderHalfSnake); 8192^3 data-parallel 128x128 65.7 / 67.5. The persistent kernels with the
// cp.async loader take kOrderColumnSnake too: with kOrderHalfSnake they spill registers.
enum InnerOrder : int {
    // column chunk q outer, rows inner, the row order reversed on every other chunk
    kOrderColumnSnake = 0,
    // column chunk q, then its two column pairs, then rows, reversed on every other pair
    kOrderHalfSnake = 1,
};

// One k-tile (32 k-steps) of outer products for one thread's 8 x 16 tile.
//   a_base: sA + (wm0 + tr) * 32, row r of the thread tile is 8 * r rows further (256 floats).
//   b_base: sB + wn0 + 4 * tc, chunk q of the thread tile is 16 * q floats further.
// KG_UNROLL < 8 keeps the k loop rolled (compact code for latency-bound launches).
template <int BN, int ORDER, int KG_UNROLL = BK / 4>
__device__ __forceinline__ void compute_ktile(const float *__restrict__ a_base, int tr,
                                              const float *__restrict__ b_base,
                                              float2 (&acc)[8][8]) {
#pragma unroll KG_UNROLL
    for (int kg = 0; kg < BK / 4; ++kg) {
        float4 a[8];
        const int achunk = (kg ^ tr) << 2;
#pragma unroll
        for (int r = 0; r < 8; ++r)
            a[r] = *reinterpret_cast<const float4 *>(a_base + r * 256 + achunk);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            float4 b[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                b[q] = *reinterpret_cast<const float4 *>(b_base + (kg * 4 + kk) * BN + 16 * q);
            auto a_pair = [&](int r) {
                const float av = kk == 0 ? a[r].x : kk == 1 ? a[r].y : kk == 2 ? a[r].z : a[r].w;
                return make_float2(av, av);
            };
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (ORDER == kOrderColumnSnake) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = (q & 1) ? 7 - i : i;
                        const float2 a2 = a_pair(r);
                        acc[r][2 * q] = __ffma2_rn(a2, make_float2(b[q].x, b[q].y), acc[r][2 * q]);
                        acc[r][2 * q + 1] =
                            __ffma2_rn(a2, make_float2(b[q].z, b[q].w), acc[r][2 * q + 1]);
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float2 bp = h == 0 ? make_float2(b[q].x, b[q].y)
                                                 : make_float2(b[q].z, b[q].w);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int r = h ? 7 - i : i;
                            acc[r][2 * q + h] = __ffma2_rn(a_pair(r), bp, acc[r][2 * q + h]);
                        }
                    }
                }
            }
        }
    }
}

// cp.async fill of one stage: A tile (BM x 32, swizzled rows) and B tile (32 x BN).
// AV / BV: 1 or 0 fixes at compile time whether A / B take 16-byte copies (only that form's
// code is emitted); -1 reads p.a_vec4 / p.b_vec4.
template <int BM, int BN, int THREADS, int AV = -1, int BV = -1>
__device__ __forceinline__ void cp_async_stage(float *sA, float *sB, const KParams &p,
                                               const float *Ab, const float *Bb, int m0, int n0,
                                               int k0, int tid) {
    if (AV < 0 ? p.a_vec4 != 0 : AV != 0) {
#pragma unroll 4
        for (int c = tid; c < BM * (BK / 4); c += THREADS) {
            const int m = c >> 3, kc = c & 7;
            const int gm = m0 + m, gk = k0 + kc * 4;
            uint32_t bytes = 0;
            const float *src = Ab;
            if (gm < p.M && gk < p.K) {
                bytes = static_cast<uint32_t>(min(4, p.K - gk)) * 4u;
                src = Ab + static_cast<long long>(gm) * p.lda + gk;
            }
            cp_async_16(smem_addr(sA + m * BK + ((kc ^ (m & 7)) << 2)), src, bytes);
        }
    } else {
#pragma unroll 4
        for (int e = tid; e < BM * BK; e += THREADS) {
            const int m = e >> 5, k = e & 31;
            const int gm = m0 + m, gk = k0 + k;
            uint32_t bytes = 0;
            const float *src = Ab;
            if (gm < p.M && gk < p.K) {
                bytes = 4u;
                src = Ab + static_cast<long long>(gm) * p.lda + gk;
            }
            cp_async_4(smem_addr(sA + m * BK + (((k >> 2) ^ (m & 7)) << 2) + (k & 3)), src, bytes);
        }
    }
    if (BV < 0 ? p.b_vec4 != 0 : BV != 0) {
#pragma unroll 4
        for (int c = tid; c < BK * (BN / 4); c += THREADS) {
            const int k = c / (BN / 4), nc = c % (BN / 4);
            const int gk = k0 + k, gn = n0 + nc * 4;
            uint32_t bytes = 0;
            const float *src = Bb;
            if (gk < p.K && gn < p.N) {
                bytes = static_cast<uint32_t>(min(4, p.N - gn)) * 4u;
                src = Bb + static_cast<long long>(gk) * p.ldb + gn;
            }
            cp_async_16(smem_addr(sB + k * BN + nc * 4), src, bytes);
        }
    } else {
#pragma unroll 4
        for (int e = tid; e < BK * BN; e += THREADS) {
            const int k = e / BN, n = e % BN;
            const int gk = k0 + k, gn = n0 + n;
            uint32_t bytes = 0;
            const float *src = Bb;
            if (gk < p.K && gn < p.N) {
                bytes = 4u;
                src = Bb + static_cast<long long>(gk) * p.ldb + gn;
            }
            cp_async_4(smem_addr(sB + k * BN + n), src, bytes);
        }
    }
}

// alpha * acc + beta * C for the thread's 8 x 16 cells (rows tr + 8r, cols 16q + 4tc + e);
// with a bias or an activation, the fused form act(alpha * acc + bias) + beta * C. Only the
// thread-tile rows r in [r_begin, r_end) are written.
// When beta != 0, C values are loaded ahead of the stores they feed: a store to C may alias a
// later load as far as the compiler knows, so interleaving them would cost one memory round
// trip per value. The plain form loads CHUNKS 4-column chunks at a time, the fused form (whose
// activation needs registers of its own) one chunk at a time; more at once spills registers
// in the persistent kernels.
// With beta != 0, asks L2 to fetch the C values the thread's epilogue will read (its 8 rows x
// 16 columns, valid addresses only), so that the epilogue's loads hit L2 instead of waiting on
// DRAM. Issued just before the epilogue (and the stream-K fix-up): the prefetches are
// fire-and-forget, so the epilogue's load rounds after the first find their lines already on
// the way. A prefetch is a hint and changes no value.
__device__ __forceinline__ void prefetch_c(const KParams &p, const float *Cb, int row0, int col0) {
    if (p.beta == 0.0f) return;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int gm = row0 + 8 * r;
        if (gm >= p.M) continue;
        const float *crow = Cb + static_cast<long long>(gm) * p.ldc;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int gn = col0 + 16 * q;
            if (gn < p.N)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(crow + gn) : "memory");
        }
    }
}

__device__ __forceinline__ void load_c4(const KParams &p, const float *crow, int gn, float (&c)[4]) {
    if (p.c_vec4 && gn + 3 < p.N) {
        const float4 v = *reinterpret_cast<const float4 *>(crow + gn);
        c[0] = v.x;
        c[1] = v.y;
        c[2] = v.z;
        c[3] = v.w;
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) c[e] = gn + e < p.N ? crow[gn + e] : 0.0f;
    }
}

__device__ __forceinline__ void store_c4(const KParams &p, float *crow, int gn, const float (&o)[4]) {
    if (p.c_vec4 && gn + 3 < p.N) {
        *reinterpret_cast<float4 *>(crow + gn) = make_float4(o[0], o[1], o[2], o[3]);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (gn + e < p.N) crow[gn + e] = o[e];
    }
}

// CHUNKS: 4-column chunks of C loaded per round trip by the plain form (2, or 1 where the
// kernel has no registers to spare). FUSED: 1 or 0 fixes the form at compile time (only its code
// is emitted); -1 decides from p.bias and p.act.
template <int CHUNKS = 2, int FUSED = -1>
__device__ __forceinline__ void epilogue(const KParams &p, float *Cb, int row0, int col0,
                                         const float2 (&acc)[8][8], int r_begin = 0,
                                         int r_end = 8) {
    static_assert(CHUNKS == 1 || CHUNKS == 2, "one or two chunks per round trip");
    const float alpha = p.alpha, beta = p.beta;
    const bool fused = FUSED < 0 ? (p.bias != nullptr || p.act != kActNone) : FUSED != 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int gm = row0 + 8 * r;
        if (r < r_begin || r >= r_end || gm >= p.M) continue;
        float *crow = Cb + static_cast<long long>(gm) * p.ldc;
        if (fused) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int gn = col0 + 16 * q;
                const float v[4] = {acc[r][2 * q].x, acc[r][2 * q].y, acc[r][2 * q + 1].x,
                                    acc[r][2 * q + 1].y};
                float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (beta != 0.0f) load_c4(p, crow, gn, c);
                float o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[e] = epilogue_apply(v[e], alpha, beta, p.bias, gn + e, p.act, c[e]);
                store_c4(p, crow, gn, o);
            }
        } else if (beta != 0.0f) {
#pragma unroll
            for (int h = 0; h < 4; h += CHUNKS) {
                float c[CHUNKS][4];
#pragma unroll
                for (int q = 0; q < CHUNKS; ++q) load_c4(p, crow, col0 + 16 * (h + q), c[q]);
#pragma unroll
                for (int q = 0; q < CHUNKS; ++q) {
                    const int qq = h + q;
                    const float o[4] = {fmaf(alpha, acc[r][2 * qq].x, beta * c[q][0]),
                                        fmaf(alpha, acc[r][2 * qq].y, beta * c[q][1]),
                                        fmaf(alpha, acc[r][2 * qq + 1].x, beta * c[q][2]),
                                        fmaf(alpha, acc[r][2 * qq + 1].y, beta * c[q][3])};
                    store_c4(p, crow, col0 + 16 * qq, o);
                }
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float o[4] = {alpha * acc[r][2 * q].x, alpha * acc[r][2 * q].y,
                                    alpha * acc[r][2 * q + 1].x, alpha * acc[r][2 * q + 1].y};
                store_c4(p, crow, col0 + 16 * q, o);
            }
        }
    }
}

template <int BM, int BN, int WARPS_M, int WARPS_N, int STAGES, int LOADER>
__global__ void __launch_bounds__(WARPS_M *WARPS_N * 32, 1)
    simt_gemm_kernel(const __grid_constant__ CUtensorMap mapA,
                     const __grid_constant__ CUtensorMap mapB, const KParams p) {
    constexpr int THREADS = WARPS_M * WARPS_N * 32;
    static_assert(BM == WARPS_M * 64 && BN == WARPS_N * 64, "64 x 64 warp tiles");
    constexpr int A_FLOATS = BM * BK;
    constexpr int STAGE_FLOATS = A_FLOATS + BK * BN;
    constexpr uint32_t STAGE_BYTES = STAGE_FLOATS * 4;

    extern __shared__ uint8_t smem_raw[];
    // The 128-byte swizzle pattern repeats every 1024 bytes of shared address space.
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    float *smem = reinterpret_cast<float *>(smem_raw + pad);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_FLOATS);
    __shared__ int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm0 = (warp / WARPS_N) * 64, wn0 = (warp % WARPS_N) * 64;
    const int tr = lane >> 2, tc = lane & 3;

    int tm, tn;
    tile_coords(blockIdx.x, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    const int m0 = tm * BM, n0 = tn * BN;
    const int KT = (p.K + BK - 1) / BK;

    if (tid == 0) {
        s_abort = 0;
        if (LOADER == kLoaderTma) {
            tma_prefetch_desc(&mapA);
            tma_prefetch_desc(&mapB);
#pragma unroll
            for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
            mbar_init_fence();
        }
    }
    __syncthreads();

    int issued = 0, consumed = 0;  // TMA k-tiles over the whole batch loop (ring position)
    for (int b = blockIdx.y; b < p.batch; b += gridDim.y) {
        float2 acc[8][8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[r][j] = make_float2(0.0f, 0.0f);

        if (LOADER == kLoaderTma) {
            auto issue = [&](int kt) {
                const int s = issued % STAGES;
                float *sA = smem + s * STAGE_FLOATS;
                mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                tma_load_3d(sA, &mapA, &full[s], kt * BK, m0, b);
                tma_load_3d(sA + A_FLOATS, &mapB, &full[s], n0, kt * BK, b);
                ++issued;
            };
            if (tid == 0)
                for (int kt = 0; kt < STAGES && kt < KT; ++kt) issue(kt);
            else
                issued += min(STAGES, KT);
            for (int kt = 0; kt < KT; ++kt) {
                const int s = consumed % STAGES;
                if (!mbar_wait(&full[s], (consumed / STAGES) & 1)) s_abort = 1;
                const float *sA = smem + s * STAGE_FLOATS;
                compute_ktile<BN, kOrderHalfSnake>(sA + (wm0 + tr) * BK, tr,
                                                   sA + A_FLOATS + wn0 + 4 * tc, acc);
                ++consumed;
                __syncthreads();  // every warp is done reading stage s
                if (s_abort) break;
                if (kt + STAGES < KT) {
                    if (tid == 0)
                        issue(kt + STAGES);
                    else
                        ++issued;
                }
            }
        } else {
            const float *Ab = p.A + static_cast<long long>(b) * p.sA;
            const float *Bb = p.B + static_cast<long long>(b) * p.sB;
#pragma unroll
            for (int s = 0; s < STAGES - 1; ++s) {
                if (s < KT) {
                    float *sA = smem + s * STAGE_FLOATS;
                    cp_async_stage<BM, BN, THREADS>(sA, sA + A_FLOATS, p, Ab, Bb, m0, n0, s * BK,
                                                    tid);
                }
                cp_async_commit();
            }
            for (int kt = 0; kt < KT; ++kt) {
                cp_async_wait<STAGES - 2>();
                __syncthreads();  // stage kt landed for all threads; stage kt - 1 is free
                const int nk = kt + STAGES - 1;
                if (nk < KT) {
                    float *sN = smem + (nk % STAGES) * STAGE_FLOATS;
                    cp_async_stage<BM, BN, THREADS>(sN, sN + A_FLOATS, p, Ab, Bb, m0, n0,
                                                    nk * BK, tid);
                }
                cp_async_commit();
                const float *sA = smem + (kt % STAGES) * STAGE_FLOATS;
                compute_ktile<BN, kOrderHalfSnake>(sA + (wm0 + tr) * BK, tr,
                                                   sA + A_FLOATS + wn0 + 4 * tc, acc);
            }
            cp_async_wait<0>();
            __syncthreads();
        }
        if (s_abort) break;
        prefetch_c(p, p.C + static_cast<long long>(b) * p.sC, m0 + wm0 + tr, n0 + wn0 + 4 * tc);
        epilogue(p, p.C + static_cast<long long>(b) * p.sC, m0 + wm0 + tr, n0 + wn0 + 4 * tc, acc);
    }

    if (LOADER == kLoaderTma && s_abort && tid == 0) {
        // Let copies already in flight land before the CTA's shared memory is released.
        for (; consumed < issued; ++consumed)
            if (!mbar_wait(&full[consumed % STAGES], (consumed / STAGES) & 1)) break;
    }
}

// ---- persistent kernel with a stream-K tail -------------------------------------------------
//
// Thread 0 issues the TMA loads of every k-tile the CTA will consume across all of its output
// tiles, STAGES - 1 k-tiles ahead of the compute (the ring does not drain between tiles).
// The grid is persistent (as many CTAs as fit on the SMs at once). Output tiles
// [0, dp_tiles) are dealt round-robin whole; the remaining tiles' k-iterations are split into
// one contiguous range per CTA (stream-K), so every CTA does the same number of k-iterations
// and no partial wave is left idle.
//
// A tile cut by a range boundary is finished by the CTA whose range holds the tile's last
// k-iteration (its "owner"); every other CTA that worked on the tile stores its fp32 partial
// sums in its own workspace slot and publishes them with a per-warp flag (release / acquire,
// value = this launch's epoch). Each CTA walks its own range backwards, so the pieces it hands
// to a higher-numbered owner are computed first and the piece it owns (whose contributors
// are lower-numbered CTAs) last: owners wait only on lower-numbered CTAs, which are resident
// or finished. Thread t of an owner warp reads exactly the partials thread t of the same warp
// of the contributing CTA wrote, so no cross-warp synchronisation is needed. The sum over
// pieces runs in a fixed order: results are deterministic.

struct PParams {
    KParams k;
    int KT;               // k-tiles per output tile
    int tiles_per_batch;  // tiles_m * tiles_n
    int dp_tiles;         // tiles done whole in the data-parallel phase
    int G;                // CTAs in the persistent grid
    long long sk_base;    // stream-K k-iterations per CTA (the first sk_rem CTAs do one more)
    int sk_rem;
    float4 *ws;           // partial sums: [G][consumer warps][32][32] float4
    unsigned int *flags;  // [G][consumer warps]
    unsigned int epoch;   // this launch's flag value (never 0)
    int chain;            // 1: wait for the kernel before (programmatic launch), 2: let the next start
};

struct Segment {
    int tile, k0, k1;
};

// The ordered list of segments (tile, k-range) CTA `c` processes: its data-parallel tiles,
// then its stream-K range from the last tile backwards. Only the cursor lives here; the
// launch constants are read from the kernel parameters at each step, so the cursor costs the
// hot loop few registers.
struct SegmentWalker {
    int t;                  // next data-parallel tile
    long long s, cur_end;   // stream-K range still to walk: [s, cur_end)

    SegmentWalker() = default;

    __device__ void init(const PParams &p, int c) {
        t = c;
        const long long base = static_cast<long long>(p.dp_tiles) * p.KT;
        s = base + c * p.sk_base + min(c, p.sk_rem);
        cur_end = s + p.sk_base + (c < p.sk_rem ? 1 : 0);
    }

    __device__ bool next(const PParams &p, Segment &seg) {
        if (t < p.dp_tiles) {
            seg.tile = t;
            seg.k0 = 0;
            seg.k1 = p.KT;
            t += p.G;
            return true;
        }
        if (cur_end <= s) return false;
        const long long tile = (cur_end - 1) / p.KT;
        const long long tb = tile * p.KT;
        const long long lo = s > tb ? s : tb;
        seg.tile = static_cast<int>(tile);
        seg.k0 = static_cast<int>(lo - tb);
        seg.k1 = static_cast<int>(cur_end - tb);
        cur_end = lo;
        return true;
    }
};

__device__ __forceinline__ long long sk_start(const PParams &p, int c) {
    return static_cast<long long>(p.dp_tiles) * p.KT + c * p.sk_base + min(c, p.sk_rem);
}

__device__ __forceinline__ void tile_origin(const PParams &p, int tile, int BM_, int BN_, int &b,
                                            int &m0, int &n0) {
    b = tile / p.tiles_per_batch;
    int tm, tn;
    tile_coords(tile - b * p.tiles_per_batch, p.k.tiles_m, p.k.tiles_n, p.k.group_m, tm, tn);
    m0 = tm * BM_;
    n0 = tn * BN_;
}

__device__ __forceinline__ void st_release_gpu(unsigned int *p, unsigned int v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Spins (bounded by kWaitLimitNs) until *flag == value. Returns false on timeout.
__device__ __forceinline__ bool wait_flag(const unsigned int *flag, unsigned int value) {
    if (ld_acquire_gpu(flag) == value) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (ld_acquire_gpu(flag) == value) return true;
        if ((spin & 15u) == 0u) {
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                raise_fault(kFaultTimeout);
                return false;
            }
            __nanosleep(64);
        }
    }
}

// Streams the k-tiles of a CTA's segment list into the shared-memory ring. With the TMA
// loader it lives in shared memory and only thread 0 touches it, so its state occupies no
// registers in the compute loop; the cp.async loader keeps one copy per thread.
struct TmaProducer {
    SegmentWalker walk;
    Segment seg;
    int kt, b, m0, n0;
    int issued;  // k-tiles issued so far (ring position)
    bool live;

    TmaProducer() = default;

    __device__ void init(const PParams &p, int c) {
        walk.init(p, c);
        kt = b = m0 = n0 = issued = 0;
        live = walk.next(p, seg);
        kt = seg.k0;
    }

    template <int BM, int BN>
    __device__ bool next(const PParams &p) {
        while (live && kt >= seg.k1) {
            live = walk.next(p, seg);
            kt = seg.k0;
        }
        if (!live) return false;
        if (kt == seg.k0) tile_origin(p, seg.tile, BM, BN, b, m0, n0);
        return true;
    }
};

// MAXREG caps registers per thread (255 leaves room for two four-warp CTAs per SM).
// KSUB: 32-wide k sub-tiles per pipeline stage (a stage then covers 32 * KSUB values of k,
// with one CTA barrier and one TMA refill per stage); the TMA loader only for KSUB > 1.
// KTAIL (KSUB > 1): the instance for K whose last stage holds padding past its first 32-wide
// sub-tile; that stage computes only the sub-tiles that hold values of k (the rest are the
// zeros TMA filled in). A separate instance, so the main loop of every other K keeps no
// branch (the branch cost 0.65% at 4096^3).
template <int BM, int BN, int WARPS_M, int WARPS_N, int STAGES, int MAXREG,
          int LOADER = kLoaderTma, int KSUB = 1, int KTAIL = 0>
__global__ void __launch_bounds__(WARPS_M *WARPS_N * 32) __maxnreg__(MAXREG)
    simt_gemm_persistent_kernel(const __grid_constant__ CUtensorMap mapA,
                                const __grid_constant__ CUtensorMap mapB, const PParams p) {
    constexpr int WARPS = WARPS_M * WARPS_N;
    static_assert(BM == WARPS_M * 64 && BN == WARPS_N * 64, "64 x 64 warp tiles");
    static_assert(STAGES >= 2, "at least double buffering");
    static_assert(KSUB == 1 || LOADER == kLoaderTma, "wide stages with the TMA loader only");
    constexpr int A_SUB = BM * BK;          // one 32-wide A sub-tile
    constexpr int A_FLOATS = KSUB * A_SUB;  // B follows the A sub-tiles
    constexpr int STAGE_FLOATS = A_FLOATS + KSUB * BK * BN;
    constexpr uint32_t STAGE_BYTES = STAGE_FLOATS * 4;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    float *smem = reinterpret_cast<float *>(smem_raw + pad);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_FLOATS);
    __shared__ int s_abort;
    __shared__ TmaProducer s_prod;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cta = blockIdx.x;

    if (tid == 0) {
        s_abort = 0;
        if (LOADER == kLoaderTma) {
            tma_prefetch_desc(&mapA);
            tma_prefetch_desc(&mapB);
#pragma unroll
            for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
            mbar_init_fence();
        }
    }

    // TMA: thread 0 streams the k-tiles of the CTA's whole segment list into the ring, the
    // first STAGES up front, then one refill into the stage just released after every k-tile.
    // cp.async: every thread walks the same cursor and copies its share of each k-tile; the
    // first STAGES - 1 up front, then, after the barrier that ends k-tile i - 1, k-tile
    // i + STAGES - 1 into the stage k-tile i - 1 used.
    TmaProducer prod_local;
    TmaProducer &prod = LOADER == kLoaderTma ? s_prod : prod_local;
    if (LOADER != kLoaderTma || tid == 0) prod.init(p, cta);
    // Launched as a programmatic dependent (the repacking kernel before it), the prologue above
    // overlapped that kernel's tail; nothing below reads global memory before it has completed.
    // The kernel after this one (the staged-C pass) may begin its launch now: it waits in the
    // same way.
    if (p.chain & 1) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (p.chain & 2) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();
    auto produce = [&]() {
        const int s = prod.issued % STAGES;
        float *sA = smem + s * STAGE_FLOATS;
        if (LOADER == kLoaderTma) {
            mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
#pragma unroll
            for (int j = 0; j < KSUB; ++j)
                tma_load_3d(sA + j * A_SUB, &mapA, &full[s], (prod.kt * KSUB + j) * BK, prod.m0,
                            prod.b);
            tma_load_3d(sA + A_FLOATS, &mapB, &full[s], prod.n0, prod.kt * KSUB * BK, prod.b);
        } else {
            cp_async_stage<BM, BN, WARPS * 32>(
                sA, sA + A_FLOATS, p.k, p.k.A + static_cast<long long>(prod.b) * p.k.sA,
                p.k.B + static_cast<long long>(prod.b) * p.k.sB, prod.m0, prod.n0, prod.kt * BK,
                tid);
        }
        ++prod.kt;
        ++prod.issued;
    };
    if (LOADER == kLoaderTma) {
        if (tid == 0)
            while (prod.issued < STAGES && prod.template next<BM, BN>(p)) produce();
    } else {
        for (int s = 0; s < STAGES - 1; ++s) {
            if (prod.template next<BM, BN>(p)) produce();
            cp_async_commit();
        }
    }

    const int wm0 = (warp / WARPS_N) * 64, wn0 = (warp % WARPS_N) * 64;
    const int tr = lane >> 2, tc = lane & 3;
    SegmentWalker walk;
    walk.init(p, cta);
    Segment seg;
    int i = 0;
    while (walk.next(p, seg)) {
        int b, m0, n0;
        tile_origin(p, seg.tile, BM, BN, b, m0, n0);
        float2 acc[8][8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[r][j] = make_float2(0.0f, 0.0f);

        for (int kt = seg.k0; kt < seg.k1; ++kt, ++i) {
            const int s = i % STAGES;
            if (LOADER == kLoaderTma) {
                if (!mbar_wait(&full[s], (i / STAGES) & 1)) s_abort = 1;
            } else {
                cp_async_wait<STAGES - 2>();
                __syncthreads();  // k-tile i landed for all threads; k-tile i - 1's stage is free
                if (prod.template next<BM, BN>(p)) produce();
                cp_async_commit();
            }
            const float *sA = smem + s * STAGE_FLOATS;
#pragma unroll
            for (int j = 0; j < KSUB; ++j) {
                if (KTAIL && j > 0 && kt == p.KT - 1 && p.k.K - kt * (KSUB * BK) <= j * BK) break;
                compute_ktile<BN, (KSUB == 2 || LOADER != kLoaderTma) ? kOrderColumnSnake
                                                                      : kOrderHalfSnake>(
                    sA + j * A_SUB + (wm0 + tr) * BK, tr, sA + A_FLOATS + j * BK * BN + wn0 + 4 * tc,
                    acc);
            }
            if (LOADER == kLoaderTma) {
                __syncthreads();  // every warp is done with stage s
                if (s_abort) break;
                if (tid == 0 && prod.template next<BM, BN>(p)) produce();
            }
        }
        if (s_abort) break;

        if (seg.k1 < p.KT) {
            // Not the owner: publish the partial sums of this piece.
            float4 *slot = p.ws + (static_cast<size_t>(cta) * WARPS + warp) * 1024;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int r = j >> 2, q = j & 3;
                slot[j * 32 + lane] = make_float4(acc[r][2 * q].x, acc[r][2 * q].y,
                                                  acc[r][2 * q + 1].x, acc[r][2 * q + 1].y);
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release_gpu(&p.flags[cta * WARPS + warp], p.epoch);
            continue;
        }
        // This CTA finishes the tile: start C's way into L2 while the fix-up (if any) runs, so
        // the epilogue's load rounds after the first find their lines arriving.
        prefetch_c(p.k, p.k.C + static_cast<long long>(b) * p.k.sC, m0 + wm0 + tr,
                   n0 + wn0 + 4 * tc);
        if (seg.k0 > 0) {
            // Owner of a split tile: add the pieces of the lower-numbered CTAs that hold
            // k-iterations [0, k0) of this tile, highest-numbered (latest k) first.
            const long long tile_begin = static_cast<long long>(seg.tile) * p.KT;
            for (int c = cta - 1; c >= 0; --c) {
                if (sk_start(p, c + 1) <= tile_begin) break;  // c's range ends before the tile
                int ok = 1;
                if (lane == 0) ok = wait_flag(&p.flags[c * WARPS + warp], p.epoch);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                const float4 *slot = p.ws + (static_cast<size_t>(c) * WARPS + warp) * 1024;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int r = j >> 2, q = j & 3;
                    const float4 v = __ldcg(slot + j * 32 + lane);
                    acc[r][2 * q].x += v.x;
                    acc[r][2 * q].y += v.y;
                    acc[r][2 * q + 1].x += v.z;
                    acc[r][2 * q + 1].y += v.w;
                }
                if (sk_start(p, c) <= tile_begin) break;  // c started this tile: last piece
            }
            // If a contributor never published (its bounded wait expired), the tile is written
            // without that piece: the output is undefined and the fault word reports it.
        }
        epilogue<LOADER == kLoaderTma ? 2 : 1>(p.k, p.k.C + static_cast<long long>(b) * p.k.sC,
                                              m0 + wm0 + tr, n0 + wn0 + 4 * tc, acc);
    }

    if (LOADER != kLoaderTma) cp_async_wait<0>();
    if (LOADER == kLoaderTma && s_abort && tid == 0) {
        // Let copies already in flight land before the CTA's shared memory is released.
        for (; i < prod.issued; ++i)
            if (!mbar_wait(&full[i % STAGES], (i / STAGES) & 1)) break;
    }
}

// ---- split-K over a thread-block cluster (grids of under one wave) ---------------------------
//
// Each output tile is computed by one cluster of S CTAs (S = 1, 2, 4 or 8) that split its
// k-tiles into S contiguous ranges of equal length (to within one), CTA rank r taking the r-th.
// After its main loop every CTA writes its fp32 accumulators into its own shared memory (the
// ring is idle by then) in fragment order: one float4 per (warp, j, lane), j = 4 * row + chunk of
// the thread's 8 x 16 tile. After a cluster barrier, CTA r adds rows [8r / S, 8(r + 1) / S) of
// every thread's tile over the S CTAs in rank order, reading the other CTAs' shared memory through
// distributed shared memory, and writes those rows of C with the epilogue. The fix-up is spread
// over all S CTAs, touches no global memory and spins on nothing; the sum runs in a fixed order,
// so results are deterministic. A second cluster barrier keeps every CTA's shared memory alive
// until the others have read it. Every CTA reaches both barriers, also after a timed-out wait.

struct CParams {
    KParams k;
    int S;   // CTAs per cluster = K slices per output tile
    int KT;  // k-tiles of the stage width per output tile
};

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared-memory address of the same location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

template <int BM, int BN, int WARPS_M, int WARPS_N, int STAGES, int KSUB>
__global__ void __launch_bounds__(WARPS_M *WARPS_N * 32, 1)
    simt_gemm_clusterk_kernel(const __grid_constant__ CUtensorMap mapA,
                              const __grid_constant__ CUtensorMap mapB, const CParams cp) {
    constexpr int WARPS = WARPS_M * WARPS_N;
    static_assert(BM == WARPS_M * 64 && BN == WARPS_N * 64, "64 x 64 warp tiles");
    constexpr int A_SUB = BM * BK;
    constexpr int A_FLOATS = KSUB * A_SUB;
    constexpr int STAGE_FLOATS = A_FLOATS + KSUB * BK * BN;
    constexpr uint32_t STAGE_BYTES = STAGE_FLOATS * 4;
    static_assert(STAGES * STAGE_FLOATS >= WARPS * 32 * 32 * 4, "partial sums fit in the ring");
    const KParams &p = cp.k;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    float *smem = reinterpret_cast<float *>(smem_raw + pad);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_FLOATS);
    __shared__ int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm0 = (warp / WARPS_N) * 64, wn0 = (warp % WARPS_N) * 64;
    const int tr = lane >> 2, tc = lane & 3;
    const int S = cp.S;
    const int rank = static_cast<int>(cluster_ctarank());
    const int tile = blockIdx.x / S;
    const int tiles_per_batch = p.tiles_m * p.tiles_n;
    const int b = tile / tiles_per_batch;
    int tm, tn;
    tile_coords(tile - b * tiles_per_batch, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    const int m0 = tm * BM, n0 = tn * BN;
    const int kt0 = static_cast<int>(static_cast<long long>(rank) * cp.KT / S);
    const int kt1 = static_cast<int>(static_cast<long long>(rank + 1) * cp.KT / S);

    if (tid == 0) {
        s_abort = 0;
        tma_prefetch_desc(&mapA);
        tma_prefetch_desc(&mapB);
#pragma unroll
        for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
        mbar_init_fence();
    }
    __syncthreads();

    float2 acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[r][j] = make_float2(0.0f, 0.0f);

    int issued = 0, consumed = 0;
    auto issue = [&](int kt) {
        const int s = issued % STAGES;
        float *sA = smem + s * STAGE_FLOATS;
        mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
#pragma unroll
        for (int j = 0; j < KSUB; ++j)
            tma_load_3d(sA + j * A_SUB, &mapA, &full[s], (kt * KSUB + j) * BK, m0, b);
        tma_load_3d(sA + A_FLOATS, &mapB, &full[s], n0, kt * KSUB * BK, b);
        ++issued;
    };
    if (tid == 0)
        for (int kt = kt0; kt < kt1 && kt < kt0 + STAGES; ++kt) issue(kt);
    else
        issued += min(STAGES, kt1 - kt0);
    for (int kt = kt0; kt < kt1; ++kt) {
        const int s = consumed % STAGES;
        if (!mbar_wait(&full[s], (consumed / STAGES) & 1)) s_abort = 1;
        const float *sA = smem + s * STAGE_FLOATS;
#pragma unroll
        for (int j = 0; j < KSUB; ++j)
            compute_ktile<BN, KSUB == 2 ? kOrderColumnSnake : kOrderHalfSnake>(
                sA + j * A_SUB + (wm0 + tr) * BK, tr, sA + A_FLOATS + j * BK * BN + wn0 + 4 * tc,
                acc);
        ++consumed;
        __syncthreads();  // every warp is done reading stage s
        if (s_abort) break;
        if (kt + STAGES < kt1) {
            if (tid == 0)
                issue(kt + STAGES);
            else
                ++issued;
        }
    }
    const bool aborted = s_abort != 0;
    if (aborted) {
        // Let copies already in flight land before the ring is reused or released.
        if (tid == 0)
            for (; consumed < issued; ++consumed)
                if (!mbar_wait(&full[consumed % STAGES], (consumed / STAGES) & 1)) break;
        __syncthreads();
    }

    // Partial sums into this CTA's own shared memory (the ring is no longer read).
    float4 *part = reinterpret_cast<float4 *>(smem);
    if (!aborted) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int r = j >> 2, q = j & 3;
            part[(warp * 32 + j) * 32 + lane] = make_float4(acc[r][2 * q].x, acc[r][2 * q].y,
                                                            acc[r][2 * q + 1].x, acc[r][2 * q + 1].y);
        }
    }
    cluster_barrier();  // every CTA's partial sums are in its shared memory

    const int r0 = rank * 8 / S, r1 = (rank + 1) * 8 / S;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        if (r < r0 || r >= r1) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t local = smem_addr(part + (warp * 32 + r * 4 + q) * 32 + lane);
            float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            for (int c = 0; c < S; ++c) {  // rank order: deterministic
                const float4 v = ld_dsmem_f4(dsmem_addr(local, static_cast<uint32_t>(c)));
                sum.x += v.x;
                sum.y += v.y;
                sum.z += v.z;
                sum.w += v.w;
            }
            acc[r][2 * q] = make_float2(sum.x, sum.y);
            acc[r][2 * q + 1] = make_float2(sum.z, sum.w);
        }
    }
    if (!aborted)
        epilogue(p, p.C + static_cast<long long>(b) * p.sC, m0 + wm0 + tr, n0 + wn0 + 4 * tc, acc,
                 r0, r1);
    cluster_barrier();  // no CTA leaves while another may still read its shared memory
}

// ---- launch templates ----------------------------------------------------------------------

template <int BM, int BN, int WARPS_M, int WARPS_N, int STAGES, int LOADER>
cudaError_t launch_impl(int id, const SimtProblem &p, cudaStream_t stream, const char **detail) {
    constexpr int THREADS = WARPS_M * WARPS_N * 32;
    constexpr size_t SMEM = static_cast<size_t>(STAGES) * (BM * BK + BK * BN) * 4 +
                            STAGES * sizeof(uint64_t) + 1024;
    auto kernel = simt_gemm_kernel<BM, BN, WARPS_M, WARPS_N, STAGES, LOADER>;

    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) {
        *detail = "cudaGetDevice failed";
        return err;
    }
    static std::once_flag attr_once[kMaxDevices];
    static cudaError_t attr_err[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) {
        *detail = "device ordinal above the library's limit";
        return cudaErrorInvalidDevice;
    }
    std::call_once(attr_once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(SMEM));
    });
    if (attr_err[dev] != cudaSuccess) {
        *detail = "cudaFuncSetAttribute(max dynamic shared memory) failed";
        return attr_err[dev];
    }

    KParams kp;
    kp.M = p.M;
    kp.N = p.N;
    kp.K = p.K;
    kp.alpha = p.alpha;
    kp.beta = p.beta;
    kp.A = p.A;
    kp.B = p.B;
    kp.C = p.C;
    kp.lda = p.lda;
    kp.ldb = p.ldb;
    kp.ldc = p.ldc;
    kp.sA = p.strideA;
    kp.sB = p.strideB;
    kp.sC = p.strideC;
    kp.batch = p.batch;
    kp.tiles_m = (p.M + BM - 1) / BM;
    kp.tiles_n = (p.N + BN - 1) / BN;
    kp.group_m = 8;
    kp.a_vec4 = operand_vec4(p.A, p.lda, p.strideA, p.batch);
    kp.b_vec4 = operand_vec4(p.B, p.ldb, p.strideB, p.batch);
    kp.c_vec4 = operand_vec4(p.C, p.ldc, p.strideC, p.batch);
    kp.bias = p.bias;
    kp.act = p.act;

    CUtensorMap mapA, mapB;
    memset(&mapA, 0, sizeof(mapA));
    memset(&mapB, 0, sizeof(mapB));
    if (LOADER == kLoaderTma) {
        if (!make_map(&mapA, p.A, p.M, p.K, p.lda, p.strideA, p.batch, BM, BK, true) ||
            !make_map(&mapB, p.B, p.K, p.N, p.ldb, p.strideB, p.batch, BK, BN, false)) {
            *detail = "cuTensorMapEncodeTiled rejected an operand";
            return cudaErrorInvalidValue;
        }
    }
    const long long tiles = static_cast<long long>(kp.tiles_m) * kp.tiles_n;
    dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(p.batch < 65535 ? p.batch : 65535));
    kernel<<<grid, THREADS, SMEM, stream>>>(mapA, mapB, kp);
    err = cudaGetLastError();
    if (err != cudaSuccess) *detail = "kernel launch failed";
    (void)id;
    return err;
}

template <int BM, int BN, int WARPS_M, int WARPS_N, int STAGES, int MAXREG = 255,
          int LOADER = kLoaderTma, int KSUB = 1, int KTAIL = 0>
cudaError_t launch_persistent(int schedule, const SimtProblem &p, cudaStream_t stream,
                              const char **detail) {
    constexpr int CONSUMER_WARPS = WARPS_M * WARPS_N;
    constexpr int THREADS = CONSUMER_WARPS * 32;
    constexpr size_t SMEM = static_cast<size_t>(STAGES) * KSUB * (BM * BK + BK * BN) * 4 +
                            2 * STAGES * sizeof(uint64_t) + 1024;
    auto kernel =
        simt_gemm_persistent_kernel<BM, BN, WARPS_M, WARPS_N, STAGES, MAXREG, LOADER, KSUB, KTAIL>;

    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) {
        *detail = "cudaGetDevice failed";
        return err;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        *detail = "device ordinal above the library's limit";
        return cudaErrorInvalidDevice;
    }
    static std::once_flag attr_once[kMaxDevices];
    static cudaError_t attr_err[kMaxDevices];
    static int occupancy[kMaxDevices];
    std::call_once(attr_once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(SMEM));
        if (attr_err[dev] == cudaSuccess)
            attr_err[dev] = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occupancy[dev], kernel,
                                                                          THREADS, SMEM);
    });
    if (attr_err[dev] != cudaSuccess) {
        *detail = "kernel attribute / occupancy query failed";
        return attr_err[dev];
    }
    const int sms = device_sms(dev);
    if (sms <= 0 || occupancy[dev] <= 0) {
        *detail = "no SM can hold the persistent kernel";
        return cudaErrorInvalidConfiguration;
    }

    PParams pp;
    KParams &kp = pp.k;
    kp.M = p.M;
    kp.N = p.N;
    kp.K = p.K;
    kp.alpha = p.alpha;
    kp.beta = p.beta;
    kp.A = p.A;
    kp.B = p.B;
    kp.C = p.C;
    kp.lda = p.lda;
    kp.ldb = p.ldb;
    kp.ldc = p.ldc;
    kp.sA = p.strideA;
    kp.sB = p.strideB;
    kp.sC = p.strideC;
    kp.batch = p.batch;
    kp.tiles_m = (p.M + BM - 1) / BM;
    kp.tiles_n = (p.N + BN - 1) / BN;
    kp.group_m = 8;
    kp.a_vec4 = operand_vec4(p.A, p.lda, p.strideA, p.batch);
    kp.b_vec4 = operand_vec4(p.B, p.ldb, p.strideB, p.batch);
    kp.c_vec4 = operand_vec4(p.C, p.ldc, p.strideC, p.batch);
    kp.bias = p.bias;
    kp.act = p.act;

    const long long tiles_per_batch = static_cast<long long>(kp.tiles_m) * kp.tiles_n;
    const long long T = tiles_per_batch * p.batch;
    if (T >= 0x7fffffffLL) {
        *detail = "too many output tiles";
        return cudaErrorInvalidValue;
    }
    const int KT = (p.K + BK * KSUB - 1) / (BK * KSUB);  // k-tiles of the stage width
    const long long g_full = static_cast<long long>(sms) * occupancy[dev];
    long long dp_tiles = T, G = T < g_full ? T : g_full;
    if (schedule == kScheduleStreamK && T % g_full != 0) {
        dp_tiles = T > g_full ? (T / g_full - 1) * g_full : 0;
        const long long sk_iters = (T - dp_tiles) * KT;
        if (dp_tiles > 0) {
            G = g_full;
        } else {
            // never more CTAs than fit at once
            G = sk_iters / sk_min_iters_per_cta(KT, KSUB);
            if (G > g_full) G = g_full;
            if (G < 1) G = 1;
        }
        pp.sk_base = sk_iters / G;
        pp.sk_rem = static_cast<int>(sk_iters % G);
    } else {
        pp.sk_base = 0;
        pp.sk_rem = 0;
    }
    pp.KT = KT;
    pp.tiles_per_batch = static_cast<int>(tiles_per_batch);
    pp.dp_tiles = static_cast<int>(dp_tiles);
    pp.G = static_cast<int>(G);
    pp.ws = nullptr;
    pp.flags = nullptr;
    pp.epoch = 1;
    pp.chain = (p.pdl ? 1 : 0) | (p.pdl_next ? 2 : 0);
    if (dp_tiles < T) {
        if (G * CONSUMER_WARPS * sizeof(unsigned int) > kFlagBytes) {
            *detail = "persistent grid above the workspace's flag capacity";
            return cudaErrorInvalidConfiguration;
        }
        const size_t partial_bytes = static_cast<size_t>(G) * CONSUMER_WARPS * 1024 * sizeof(float4);
        err = workspace_for(dev, stream, partial_bytes, &pp.ws, &pp.flags, &pp.epoch);
        if (err != cudaSuccess) {
            *detail = "stream-K workspace allocation failed";
            return err;
        }
    }

    CUtensorMap mapA, mapB;
    memset(&mapA, 0, sizeof(mapA));
    memset(&mapB, 0, sizeof(mapB));
    if (LOADER == kLoaderTma &&
        (!make_map(&mapA, p.A, p.M, p.K, p.lda, p.strideA, p.batch, BM, BK, true) ||
         !make_map(&mapB, p.B, p.K, p.N, p.ldb, p.strideB, p.batch, BK * KSUB, BN, false))) {
        *detail = "cuTensorMapEncodeTiled rejected an operand";
        return cudaErrorInvalidValue;
    }
    if (const char *env = std::getenv("SGEMM_LOG"); env && *env && env[0] != '0')
        std::fprintf(stderr,
                     "[sgemm] persistent %dx%d: occupancy %d, grid %lld, tiles %lld, dp_tiles %lld, "
                     "k-tiles/tile %d, stream-K iters/CTA %lld (+1 for %d)\n",
                     BM, BN, occupancy[dev], G, T, dp_tiles, KT, pp.sk_base, pp.sk_rem);
    if (p.pdl) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(G), 1, 1);
        cfg.blockDim = dim3(THREADS, 1, 1);
        cfg.dynamicSmemBytes = SMEM;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaLaunchKernelEx(&cfg, kernel, mapA, mapB, pp);
    } else {
        kernel<<<static_cast<unsigned>(G), THREADS, SMEM, stream>>>(mapA, mapB, pp);
    }
    err = cudaGetLastError();
    if (err != cudaSuccess) *detail = "kernel launch failed";
    return err;
}

template <int BM, int BN, int WARPS_M, int WARPS_N, int STAGES, int KSUB>
cudaError_t launch_clusterk(const SimtProblem &p, cudaStream_t stream, const char **detail) {
    constexpr int THREADS = WARPS_M * WARPS_N * 32;
    constexpr size_t SMEM = static_cast<size_t>(STAGES) * KSUB * (BM * BK + BK * BN) * 4 +
                            STAGES * sizeof(uint64_t) + 1024;
    auto kernel = simt_gemm_clusterk_kernel<BM, BN, WARPS_M, WARPS_N, STAGES, KSUB>;

    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) {
        *detail = "cudaGetDevice failed";
        return err;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        *detail = "device ordinal above the library's limit";
        return cudaErrorInvalidDevice;
    }
    static std::once_flag attr_once[kMaxDevices];
    static cudaError_t attr_err[kMaxDevices];
    std::call_once(attr_once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(SMEM));
    });
    if (attr_err[dev] != cudaSuccess) {
        *detail = "cudaFuncSetAttribute(max dynamic shared memory) failed";
        return attr_err[dev];
    }
    const int sms = device_sms(dev);

    CParams cp;
    KParams &kp = cp.k;
    kp.M = p.M;
    kp.N = p.N;
    kp.K = p.K;
    kp.alpha = p.alpha;
    kp.beta = p.beta;
    kp.A = p.A;
    kp.B = p.B;
    kp.C = p.C;
    kp.lda = p.lda;
    kp.ldb = p.ldb;
    kp.ldc = p.ldc;
    kp.sA = p.strideA;
    kp.sB = p.strideB;
    kp.sC = p.strideC;
    kp.batch = p.batch;
    kp.tiles_m = (p.M + BM - 1) / BM;
    kp.tiles_n = (p.N + BN - 1) / BN;
    kp.group_m = 8;
    kp.a_vec4 = 1;
    kp.b_vec4 = 1;
    kp.c_vec4 = operand_vec4(p.C, p.ldc, p.strideC, p.batch);
    kp.bias = p.bias;
    kp.act = p.act;
    const long long tiles = static_cast<long long>(kp.tiles_m) * kp.tiles_n * p.batch;
    cp.KT = (p.K + BK * KSUB - 1) / (BK * KSUB);
    cp.S = clusterk_slices(tiles, cp.KT, sms > 0 ? sms : 1);
    if (tiles * cp.S > 0x7fffffffLL) {
        *detail = "too many output tiles for the cluster split-K grid";
        return cudaErrorInvalidValue;
    }

    CUtensorMap mapA, mapB;
    if (!make_map(&mapA, p.A, p.M, p.K, p.lda, p.strideA, p.batch, BM, BK, true) ||
        !make_map(&mapB, p.B, p.K, p.N, p.ldb, p.strideB, p.batch, BK * KSUB, BN, false)) {
        *detail = "cuTensorMapEncodeTiled rejected an operand";
        return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * cp.S), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cp.S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (const char *env = std::getenv("SGEMM_LOG"); env && *env && env[0] != '0')
        std::fprintf(stderr, "[sgemm] cluster split-K %dx%d: tiles %lld, slices %d, k-tiles %d\n",
                     BM, BN, tiles, cp.S, cp.KT);
    err = cudaLaunchKernelEx(&cfg, kernel, mapA, mapB, cp);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) *detail = "cluster split-K kernel launch failed";
    return err;
}

}  // namespace
}  // namespace sg
