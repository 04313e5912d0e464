// simt_gemm.cu: FP32 SIMT GEMM kernels for sm_103a, C = alpha * (A . B) + beta * C, row-major.
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
#include "epilogue.cuh"
#include "ptx.cuh"
#include "raster.cuh"
#include "simt_gemm.cuh"
#include "skinny_gemm.cuh"

#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

namespace sg {
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
template <int BM, int BN, int THREADS>
__device__ __forceinline__ void cp_async_stage(float *sA, float *sB, const KParams &p,
                                               const float *Ab, const float *Bb, int m0, int n0,
                                               int k0, int tid) {
    if (p.a_vec4) {
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
    if (p.b_vec4) {
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
// with a bias or an activation, the fused form act(alpha * acc + bias) + beta * C.
__device__ __forceinline__ void epilogue(const KParams &p, float *Cb, int row0, int col0,
                                         const float2 (&acc)[8][8]) {
    const float alpha = p.alpha, beta = p.beta;
    const bool fused = p.bias != nullptr || p.act != kActNone;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int gm = row0 + 8 * r;
        if (gm >= p.M) continue;
        float *crow = Cb + static_cast<long long>(gm) * p.ldc;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int gn = col0 + 16 * q;
            const float v[4] = {acc[r][2 * q].x, acc[r][2 * q].y, acc[r][2 * q + 1].x,
                                acc[r][2 * q + 1].y};
            if (fused) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (gn + e < p.N)
                        crow[gn + e] = epilogue_value(v[e], alpha, beta, p.bias, gn + e, p.act,
                                                      crow + gn + e);
            } else if (p.c_vec4 && gn + 3 < p.N) {
                float4 o;
                if (beta != 0.0f) {
                    const float4 c = *reinterpret_cast<const float4 *>(crow + gn);
                    o = make_float4(fmaf(alpha, v[0], beta * c.x), fmaf(alpha, v[1], beta * c.y),
                                    fmaf(alpha, v[2], beta * c.z), fmaf(alpha, v[3], beta * c.w));
                } else {
                    o = make_float4(alpha * v[0], alpha * v[1], alpha * v[2], alpha * v[3]);
                }
                *reinterpret_cast<float4 *>(crow + gn) = o;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (gn + e < p.N) {
                        crow[gn + e] = beta != 0.0f ? fmaf(alpha, v[e], beta * crow[gn + e])
                                                    : alpha * v[e];
                    }
                }
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
template <int BM, int BN, int WARPS_M, int WARPS_N, int STAGES, int MAXREG,
          int LOADER = kLoaderTma, int KSUB = 1>
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
            for (int j = 0; j < KSUB; ++j)
                compute_ktile<BN, (KSUB == 2 || LOADER != kLoaderTma) ? kOrderColumnSnake
                                                                      : kOrderHalfSnake>(
                    sA + j * A_SUB + (wm0 + tr) * BK, tr, sA + A_FLOATS + j * BK * BN + wn0 + 4 * tc,
                    acc);
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
        epilogue(p.k, p.k.C + static_cast<long long>(b) * p.k.sC, m0 + wm0 + tr,
                 n0 + wn0 + 4 * tc, acc);
    }

    if (LOADER != kLoaderTma) cp_async_wait<0>();
    if (LOADER == kLoaderTma && s_abort && tid == 0) {
        // Let copies already in flight land before the CTA's shared memory is released.
        for (; i < prod.issued; ++i)
            if (!mbar_wait(&full[i % STAGES], (i / STAGES) & 1)) break;
    }
}

// ---- host side ---------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

long long round_up16(long long v) { return (v + 15) / 16 * 16; }

// rows x cols fp32 matrix with leading dimension ld, `batch` copies `stride` elements apart,
// read in boxes of box_rows x box_cols.
bool make_map(CUtensorMap *map, const float *base, long long rows, long long cols, long long ld,
              long long stride, int batch, int box_rows, int box_cols, bool swizzle128) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const long long stride_bytes =
        batch > 1 ? stride * 4 : round_up16(rows * ld * 4 > 16 ? rows * ld * 4 : 16);
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 4),
                             static_cast<cuuint64_t>(stride_bytes)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

bool operand_vec4(const float *ptr, long long ld, long long stride, int batch) {
    return aligned16(ptr) && ld % 4 == 0 && (batch <= 1 || stride % 4 == 0);
}

bool tma_ok(const SimtProblem &p) {
    // TMA needs 16-byte aligned bases and byte strides; a zero batch stride (broadcast
    // operand) goes to the cp.async loader.
    if (!operand_vec4(p.A, p.lda, p.strideA, p.batch)) return false;
    if (!operand_vec4(p.B, p.ldb, p.strideB, p.batch)) return false;
    if (p.batch > 1 && (p.strideA == 0 || p.strideB == 0)) return false;
    return true;
}

const SimtConfig kConfigs[] = {
    {"dp_tma_128x256_s4", 128, 256, 2, 4, 4, kLoaderTma, kScheduleDataParallel},
    {"dp_tma_256x128_s4", 256, 128, 4, 2, 4, kLoaderTma, kScheduleDataParallel},
    {"dp_tma_128x128_s3", 128, 128, 2, 2, 3, kLoaderTma, kScheduleDataParallel},
    {"dp_cpasync_128x256_s4", 128, 256, 2, 4, 4, kLoaderCpAsync, kScheduleDataParallel},
    {"dp_cpasync_128x128_s3", 128, 128, 2, 2, 3, kLoaderCpAsync, kScheduleDataParallel},
    {"sk_tma_ws_128x256_s4", 128, 256, 2, 4, 4, kLoaderTma, kScheduleStreamK},
    {"pdp_tma_ws_128x256_s4", 128, 256, 2, 4, 4, kLoaderTma, kSchedulePersistentDP},
    {"sk_tma_ws_256x128_s4", 256, 128, 4, 2, 4, kLoaderTma, kScheduleStreamK},
    {"sk_tma_ws_128x128_s3", 128, 128, 2, 2, 3, kLoaderTma, kScheduleStreamK},
    {"sk_tma_ws_128x128_s4", 128, 128, 2, 2, 4, kLoaderTma, kScheduleStreamK},
    {"skinny_tall_n8", 0, 0, 0, 0, 0, kLoaderCpAsync, kScheduleSkinny},
    {"skinny_wide_m8", 0, 0, 0, 0, 0, kLoaderCpAsync, kScheduleSkinny},
    {"sk_cpasync_128x256_s4", 128, 256, 2, 4, 4, kLoaderCpAsync, kScheduleStreamK},
    {"sk_cpasync_256x128_s4", 256, 128, 4, 2, 4, kLoaderCpAsync, kScheduleStreamK},
    {"packed_sk_tma_128x256_s4", 128, 256, 2, 4, 4, kLoaderTma, kScheduleStreamK},
    {"packed_dp_tma_128x128_s3", 128, 128, 2, 2, 3, kLoaderTma, kScheduleDataParallel},
    {"sk_tma_ws_128x256_k64_s2", 128, 256, 2, 4, 2, kLoaderTma, kScheduleStreamK},
    {"sk_tma_ws_256x128_k64_s2", 256, 128, 4, 2, 2, kLoaderTma, kScheduleStreamK},
    {"packed_sk_tma_256x128_k64_s2", 256, 128, 4, 2, 2, kLoaderTma, kScheduleStreamK},
    {"splitk_cpasync_64x64", 64, 64, 1, 1, 2, kLoaderCpAsync, kScheduleDataParallel},
};
constexpr int kNumConfigs = sizeof(kConfigs) / sizeof(kConfigs[0]);

constexpr int kMaxDevices = 64;

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


// ---- persistent launch: workspace, grid size and the data-parallel / stream-K split ---------

struct WorkspaceEntry {
    int dev;
    cudaStream_t stream;
    void *ptr;
    size_t bytes;
    unsigned int epoch;
};
std::mutex g_ws_mutex;
std::vector<WorkspaceEntry> g_ws;

constexpr size_t kFlagBytes = 64 * 1024;  // room for 2048 CTAs x 8 warps of flags

// Workspace for (device, stream): kFlagBytes of flags, then `partial_bytes` of partial sums.
// Returns the next epoch for this workspace through `epoch`.
cudaError_t workspace_for(int dev, cudaStream_t stream, size_t partial_bytes, float4 **ws,
                          unsigned int **flags, unsigned int *epoch) {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    WorkspaceEntry *e = nullptr;
    for (auto &w : g_ws)
        if (w.dev == dev && w.stream == stream) e = &w;
    const size_t need = kFlagBytes + partial_bytes;
    if (e && e->bytes < need) {
        cudaError_t err = cudaFree(e->ptr);  // waits for work that may still use it
        e->ptr = nullptr;
        if (err != cudaSuccess) return err;
    }
    if (!e) {
        g_ws.push_back({dev, stream, nullptr, 0, 0});
        e = &g_ws.back();
    }
    if (!e->ptr) {
        cudaError_t err = cudaMalloc(&e->ptr, need);
        if (err != cudaSuccess) {
            e->ptr = nullptr;
            e->bytes = 0;
            return err;
        }
        e->bytes = need;
        e->epoch = 0;
        err = cudaMemsetAsync(e->ptr, 0, kFlagBytes, stream);
        if (err != cudaSuccess) return err;
    }
    if (++e->epoch == 0) ++e->epoch;
    *epoch = e->epoch;
    *flags = static_cast<unsigned int *>(e->ptr);
    *ws = reinterpret_cast<float4 *>(static_cast<char *>(e->ptr) + kFlagBytes);
    return cudaSuccess;
}

struct DeviceInfo {
    int sms = 0;
};

int device_sms(int dev) {
    static std::mutex mu;
    static int cache[64] = {0};
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 0;
    if (dev >= 0 && dev < 64) cache[dev] = sms;
    return sms;
}

// k-tiles per CTA when a grid of under one wave splits every tile along K. Each CTA
// computes c k-tiles; a tile's owner then adds the partial sums of the other
// ceil(KT / c) - 1 pieces, and reading one piece (64 KiB per warp, from L2) costs about a
// fifth of a 32-wide k-tile of paired FMAs, so c near sqrt(KT / (5 * KSUB)) minimises
// c + (KT / c) / (5 * KSUB). (128^3: 1 k-tile per CTA on 4 SMs instead of all 4 on one.)
int sk_min_iters_per_cta(long long KT, int KSUB) {
    int c = 1;
    while (static_cast<long long>(c + 1) * (c + 1) * 5 * KSUB <= KT) ++c;
    return c;
}

template <int BM, int BN, int WARPS_M, int WARPS_N, int STAGES, int MAXREG = 255,
          int LOADER = kLoaderTma, int KSUB = 1>
cudaError_t launch_persistent(int schedule, const SimtProblem &p, cudaStream_t stream,
                              const char **detail) {
    constexpr int CONSUMER_WARPS = WARPS_M * WARPS_N;
    constexpr int THREADS = CONSUMER_WARPS * 32;
    constexpr size_t SMEM = static_cast<size_t>(STAGES) * KSUB * (BM * BK + BK * BN) * 4 +
                            2 * STAGES * sizeof(uint64_t) + 1024;
    auto kernel =
        simt_gemm_persistent_kernel<BM, BN, WARPS_M, WARPS_N, STAGES, MAXREG, LOADER, KSUB>;

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
    kernel<<<static_cast<unsigned>(G), THREADS, SMEM, stream>>>(mapA, mapB, pp);
    err = cudaGetLastError();
    if (err != cudaSuccess) *detail = "kernel launch failed";
    return err;
}

bool packable(const SimtProblem &p);
cudaError_t launch_small_splitk(const SimtProblem &p, cudaStream_t stream, const char **detail);
cudaError_t launch_packed(int inner, const SimtProblem &p, cudaStream_t stream,
                          const char **detail);

}  // namespace

int simt_num_configs() { return kNumConfigs; }

int simt_device_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();  // leave no sticky error for the caller
        return 0;
    }
    return device_sms(dev);
}

const SimtConfig &simt_config(int id) { return kConfigs[id]; }

bool simt_config_supports(int id, const SimtProblem &p) {
    if (id < 0 || id >= kNumConfigs) return false;
    if (id == 10) return skinny_supports(kSkinnyTall, p);
    if (id == 11) return skinny_supports(kSkinnyWide, p);
    if (id == 14 || id == 15 || id == 18) return packable(p);
    if (kConfigs[id].loader == kLoaderTma) return tma_ok(p);
    return true;
}

cudaError_t simt_launch(int id, const SimtProblem &p, cudaStream_t stream, const char **detail) {
    switch (id) {
        case 0: return launch_impl<128, 256, 2, 4, 4, kLoaderTma>(id, p, stream, detail);
        case 1: return launch_impl<256, 128, 4, 2, 4, kLoaderTma>(id, p, stream, detail);
        case 2: return launch_impl<128, 128, 2, 2, 3, kLoaderTma>(id, p, stream, detail);
        case 3: return launch_impl<128, 256, 2, 4, 4, kLoaderCpAsync>(id, p, stream, detail);
        case 4: return launch_impl<128, 128, 2, 2, 3, kLoaderCpAsync>(id, p, stream, detail);
        case 5: return launch_persistent<128, 256, 2, 4, 4>(kScheduleStreamK, p, stream, detail);
        case 6: return launch_persistent<128, 256, 2, 4, 4>(kSchedulePersistentDP, p, stream, detail);
        case 7: return launch_persistent<256, 128, 4, 2, 4>(kScheduleStreamK, p, stream, detail);
        case 8: return launch_persistent<128, 128, 2, 2, 3, 255>(kScheduleStreamK, p, stream, detail);
        case 9: return launch_persistent<128, 128, 2, 2, 4, 248>(kScheduleStreamK, p, stream, detail);
        case 10: return skinny_launch(kSkinnyTall, p, stream, detail);
        case 11: return skinny_launch(kSkinnyWide, p, stream, detail);
        case 12:
            return launch_persistent<128, 256, 2, 4, 4, 255, kLoaderCpAsync>(kScheduleStreamK, p,
                                                                            stream, detail);
        case 13:
            return launch_persistent<256, 128, 4, 2, 4, 255, kLoaderCpAsync>(kScheduleStreamK, p,
                                                                            stream, detail);
        case 14: return launch_packed(5, p, stream, detail);
        case 15: return launch_packed(2, p, stream, detail);
        case 16:
            return launch_persistent<128, 256, 2, 4, 2, 255, kLoaderTma, 2>(kScheduleStreamK, p,
                                                                           stream, detail);
        case 17:
            return launch_persistent<256, 128, 4, 2, 2, 255, kLoaderTma, 2>(kScheduleStreamK, p,
                                                                           stream, detail);
        case 18: return launch_packed(17, p, stream, detail);
        case 19: return launch_small_splitk(p, stream, detail);
        default: *detail = "unknown SIMT configuration"; return cudaErrorInvalidValue;
    }
}

cudaError_t release_workspaces() {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    cudaError_t first = cudaSuccess;
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto &w : g_ws) {
        if (!w.ptr) continue;
        cudaSetDevice(w.dev);
        cudaError_t err = cudaFree(w.ptr);
        if (err != cudaSuccess && first == cudaSuccess) first = err;
    }
    cudaSetDevice(cur);
    g_ws.clear();
    return first;
}

unsigned int simt_take_fault_word(cudaStream_t stream) {
    unsigned int word = 0;
    if (cudaMemcpyFromSymbolAsync(&word, g_fault_word, sizeof(word), 0, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess)
        return 0;
    const unsigned int zero = 0;
    cudaMemcpyToSymbolAsync(g_fault_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
    cudaStreamSynchronize(stream);
    return word;
}

// ---- stream-K without any allocation: partial sums in a static device array ------------------
//
// Same kernel and schedule as configuration sk_tma_ws_128x256_s4, but the partial-sum slots and
// flags live in g_static_scratch, a file-scope device array that every device holding this
// library carries until the process exits, instead of a cudaMalloc'd workspace.
namespace {

constexpr int kStaticSlots = 160;          // persistent CTAs the array serves (152 SMs fit)
constexpr int kStaticWarps = 8;            // warps of the 128 x 256 kernel
constexpr size_t kStaticFlagFloat4 = 512;  // 8 KiB of flag words, one per warp and slot
constexpr size_t kStaticSlotFloat4 = static_cast<size_t>(kStaticWarps) * 1024;  // 128 KiB
constexpr size_t kStaticScratchFloat4 =
    kStaticFlagFloat4 + static_cast<size_t>(kStaticSlots) * kStaticSlotFloat4;  // 20 MiB + 8 KiB
static_assert(kStaticSlots * kStaticWarps * sizeof(unsigned int) <= kStaticFlagFloat4 * 16,
              "flag words must fit their region");

static __device__ __align__(256) float4 g_static_scratch[kStaticScratchFloat4];

struct StaticScratchState {
    std::once_flag once;
    void *ptr = nullptr;  // device address of g_static_scratch on this device
    int occupancy = 0;
    cudaError_t err = cudaSuccess;
};
StaticScratchState g_static_state[kMaxDevices];

thread_local char t_static_detail[160];

}  // namespace

cudaError_t simt_launch_noalloc(const SimtProblem &p, cudaStream_t stream, const char **detail) {
    constexpr int BM = 128, BN = 256, WARPS_M = 2, WARPS_N = 4, STAGES = 4, MAXREG = 255;
    constexpr int WARPS = WARPS_M * WARPS_N;
    constexpr int THREADS = WARPS * 32;
    constexpr size_t SMEM = static_cast<size_t>(STAGES) * (BM * BK + BK * BN) * 4 +
                            2 * STAGES * sizeof(uint64_t) + 1024;
    static_assert(WARPS == kStaticWarps, "slot layout follows the kernel's warp count");
    auto kernel = simt_gemm_persistent_kernel<BM, BN, WARPS_M, WARPS_N, STAGES, MAXREG>;

    if (!tma_ok(p)) {
        *detail = "needs 16-byte aligned A and B with lda and ldb multiples of 4";
        return cudaErrorNotSupported;
    }
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
    // Set-up, once per device, with that device current: the host-side name of the array is
    // not a device address, so ask the runtime for this device's copy.
    StaticScratchState &st = g_static_state[dev];
    std::call_once(st.once, [&] {
        void *ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(SMEM));
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&st.occupancy, kernel, THREADS, SMEM);
        st.ptr = ptr;
        st.err = e;
    });
    if (st.err != cudaSuccess || !st.ptr) {
        *detail = "static scratch set-up (cudaGetSymbolAddress / kernel attributes) failed";
        return st.err != cudaSuccess ? st.err : cudaErrorInvalidSymbol;
    }
    const int sms = device_sms(dev);
    if (sms <= 0 || st.occupancy <= 0) {
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
    kp.a_vec4 = 1;
    kp.b_vec4 = 1;
    kp.c_vec4 = operand_vec4(p.C, p.ldc, p.strideC, p.batch);
    kp.bias = nullptr;  // plain product only
    kp.act = 0;

    const long long tiles_per_batch = static_cast<long long>(kp.tiles_m) * kp.tiles_n;
    const long long T = tiles_per_batch * p.batch;
    if (T >= 0x7fffffffLL) {
        *detail = "too many output tiles";
        return cudaErrorInvalidValue;
    }
    const int KT = (p.K + BK - 1) / BK;
    const long long g_full = static_cast<long long>(sms) * st.occupancy;
    long long dp_tiles = T, G = T < g_full ? T : g_full;
    pp.sk_base = 0;
    pp.sk_rem = 0;
    if (T % g_full != 0) {
        dp_tiles = T > g_full ? (T / g_full - 1) * g_full : 0;
        const long long sk_iters = (T - dp_tiles) * KT;
        if (dp_tiles > 0) {
            G = g_full;
        } else {
            // never more CTAs than fit at once
            G = sk_iters / sk_min_iters_per_cta(KT, 1);
            if (G > g_full) G = g_full;
            if (G < 1) G = 1;
        }
        pp.sk_base = sk_iters / G;
        pp.sk_rem = static_cast<int>(sk_iters % G);
    }
    pp.KT = KT;
    pp.tiles_per_batch = static_cast<int>(tiles_per_batch);
    pp.dp_tiles = static_cast<int>(dp_tiles);
    pp.G = static_cast<int>(G);
    pp.ws = nullptr;
    pp.flags = nullptr;
    pp.epoch = 1;
    if (dp_tiles < T) {
        // The stream-K part needs one slot per CTA.
        if (G > kStaticSlots) {
            std::snprintf(t_static_detail, sizeof(t_static_detail),
                          "this call needs %lld partial-sum slots of 128 KiB; the static scratch "
                          "holds %d",
                          G, kStaticSlots);
            *detail = t_static_detail;
            return cudaErrorNotSupported;
        }
        pp.flags = static_cast<unsigned int *>(st.ptr);
        pp.ws = static_cast<float4 *>(st.ptr) + kStaticFlagFloat4;
        // The array keeps the previous call's flags: clear the ones this call uses.
        err = cudaMemsetAsync(pp.flags, 0, static_cast<size_t>(G) * WARPS * sizeof(unsigned int),
                              stream);
        if (err != cudaSuccess) {
            *detail = "clearing the static scratch flags failed";
            return err;
        }
    }

    CUtensorMap mapA, mapB;
    if (!make_map(&mapA, p.A, p.M, p.K, p.lda, p.strideA, p.batch, BM, BK, true) ||
        !make_map(&mapB, p.B, p.K, p.N, p.ldb, p.strideB, p.batch, BK, BN, false)) {
        *detail = "cuTensorMapEncodeTiled rejected an operand";
        return cudaErrorInvalidValue;
    }
    kernel<<<static_cast<unsigned>(G), THREADS, SMEM, stream>>>(mapA, mapB, pp);
    err = cudaGetLastError();
    if (err != cudaSuccess) *detail = "kernel launch failed";
    return err;
}

// ---- failure-path self-test: a bounded wait that can never be satisfied -----------------------
namespace {

static __device__ unsigned int g_selftest_flag;  // never written: stays 0

// which == 0: waits on an mbarrier phase no thread completes; which == 1: waits for a flag value
// nothing stores. Both waits give up after kWaitLimitNs, raise the fault word and return.
__global__ void selftest_wait_kernel(int which) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    if (which == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
        mbar_wait(&bar, 0);
    } else {
        wait_flag(&g_selftest_flag, 1u);
    }
}

}  // namespace

cudaError_t simt_selftest_wait(int which, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(which);
    return cudaGetLastError();
}

// ---- repacking operands TMA cannot read -------------------------------------------------------
//
// TMA needs 16-byte aligned rows (base and leading dimension). An operand without them is
// copied once into a workspace with its leading dimension rounded up to a multiple of 4,
// then the TMA kernels run on the copy: the copy streams the operand at HBM speed, which
// is cheaper than feeding every k-tile through 4-byte cp.async copies.
namespace {

// Rows run over the grid's y dimension (batch entries stacked), columns over threads.
__global__ void pack_rows_kernel(const float *__restrict__ src, long long lds, long long ss,
                                 float *__restrict__ dst, long long ldd, long long sd, int rows,
                                 int cols, int batch) {
    const long long nrows = static_cast<long long>(rows) * batch;
    for (long long gr = blockIdx.y; gr < nrows; gr += gridDim.y) {
        const long long b = gr / rows, r = gr - b * rows;
        const float *s = src + b * ss + r * lds;
        float *d = dst + b * sd + r * ldd;
        for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < cols; c += gridDim.x * blockDim.x)
            d[c] = s[c];
    }
}

dim3 rows_grid(long long rows, int cols) {
    const unsigned x = static_cast<unsigned>(std::min<long long>((cols + 255) / 256, 8));
    const unsigned y = static_cast<unsigned>(std::min<long long>(rows, 65535));
    return dim3(x, y);
}

struct PackWorkspace {
    int dev;
    cudaStream_t stream;
    int slot;  // 0: transposed copies, 1: realigned copies (both may live at once)
    void *ptr;
    size_t bytes;
};
std::mutex g_pack_mutex;
std::vector<PackWorkspace> g_pack_ws;

constexpr int kSlotTransposed = 0;
constexpr int kSlotRealigned = 1;
constexpr int kSlotSplitK = 2;        // split-K partial tiles
constexpr int kSlotSplitKCount = 3;   // split-K per-tile counts (zero between launches)

// *fresh (when given) reports a new allocation, whose contents are undefined.
cudaError_t pack_workspace(int dev, cudaStream_t stream, int slot, size_t bytes, float **out,
                           bool *fresh = nullptr) {
    if (fresh) *fresh = false;
    std::lock_guard<std::mutex> lock(g_pack_mutex);
    PackWorkspace *e = nullptr;
    for (auto &w : g_pack_ws)
        if (w.dev == dev && w.stream == stream && w.slot == slot) e = &w;
    if (e && e->bytes < bytes) {
        cudaError_t err = cudaFree(e->ptr);
        e->ptr = nullptr;
        e->bytes = 0;
        if (err != cudaSuccess) return err;
    }
    if (!e) {
        g_pack_ws.push_back({dev, stream, slot, nullptr, 0});
        e = &g_pack_ws.back();
    }
    if (!e->ptr) {
        cudaError_t err = cudaMalloc(&e->ptr, bytes);
        if (err != cudaSuccess) {
            e->ptr = nullptr;
            return err;
        }
        e->bytes = bytes;
        if (fresh) *fresh = true;
    }
    *out = static_cast<float *>(e->ptr);
    return cudaSuccess;
}

bool packable(const SimtProblem &p) {
    // a broadcast operand (batch stride 0) would need one copy per batch entry: not packed
    return p.batch <= 1 || (p.strideA != 0 && p.strideB != 0);
}

// ---- small problems: one warp per 64 x 64 tile, K split over CTAs ------------------------
//
// For problems of a few tiles the large kernels leave most SMs idle and spend their time on
// cold instruction fetch of a fully unrolled loop. Here each CTA is one warp computing a
// 64 x 64 tile (the same 8 x 16 thread tile and fragment layout) over a slice of K, from a
// two-stage cp.async ring (any alignment) and a rolled k loop. With more than one slice each
// CTA stores its partial tile, and the CTA that finishes a tile last (an atomic count per
// tile; nothing waits) adds the slices in slice order and applies the epilogue, so results
// do not depend on which CTA finishes when; it then resets the count for the next call.

struct SmallParams {
    KParams k;
    int split;                // K slices per tile
    int kt_per_slice;         // 32-wide k-tiles per slice
    float4 *partials;         // [tile][slice][32 x 32 float4]
    unsigned int *counters;   // [tile]: slices finished
};

constexpr int kSmallStageFloats = 64 * BK + BK * 64;

__global__ void __launch_bounds__(32) small_splitk_kernel(const SmallParams sp) {
    const KParams &p = sp.k;
    __shared__ __align__(16) float smem[2][kSmallStageFloats];
    const int lane = threadIdx.x;
    const int tile = blockIdx.x, slice = blockIdx.y;
    const int tiles_per_batch = p.tiles_m * p.tiles_n;
    const int b = tile / tiles_per_batch;
    int tm, tn;
    tile_coords(tile - b * tiles_per_batch, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    const int m0 = tm * 64, n0 = tn * 64;
    const int KT = (p.K + BK - 1) / BK;
    const int kt0 = slice * sp.kt_per_slice;
    const int kt1 = min(KT, kt0 + sp.kt_per_slice);
    const float *Ab = p.A + static_cast<long long>(b) * p.sA;
    const float *Bb = p.B + static_cast<long long>(b) * p.sB;
    const int tr = lane >> 2, tc = lane & 3;

    float2 acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[r][j] = make_float2(0.0f, 0.0f);

    if (kt0 < kt1)
        cp_async_stage<64, 64, 32>(smem[0], smem[0] + 64 * BK, p, Ab, Bb, m0, n0, kt0 * BK, lane);
    cp_async_commit();
#pragma unroll 1
    for (int kt = kt0; kt < kt1; ++kt) {
        const int s = (kt - kt0) & 1;
        if (kt + 1 < kt1)
            cp_async_stage<64, 64, 32>(smem[s ^ 1], smem[s ^ 1] + 64 * BK, p, Ab, Bb, m0, n0,
                                       (kt + 1) * BK, lane);
        cp_async_commit();
        cp_async_wait<1>();
        __syncwarp();  // k-tile kt landed for the whole warp
        compute_ktile<64, kOrderHalfSnake, 1>(smem[s] + tr * BK, tr, smem[s] + 64 * BK + 4 * tc,
                                              acc);
        __syncwarp();  // stage s is free for the load two k-tiles ahead
    }
    cp_async_wait<0>();

    float *Cb = p.C + static_cast<long long>(b) * p.sC;
    if (sp.split == 1) {
        epilogue(p, Cb, m0 + tr, n0 + 4 * tc, acc);
        return;
    }
    float4 *mine = sp.partials + (static_cast<size_t>(tile) * sp.split + slice) * 1024;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int r = j >> 2, q = j & 3;
        mine[j * 32 + lane] = make_float4(acc[r][2 * q].x, acc[r][2 * q].y, acc[r][2 * q + 1].x,
                                          acc[r][2 * q + 1].y);
    }
    __threadfence();
    __syncwarp();
    unsigned int done = 0;
    if (lane == 0) done = atomicAdd(&sp.counters[tile], 1u);
    done = __shfl_sync(0xffffffffu, done, 0);
    if (done != static_cast<unsigned int>(sp.split - 1)) return;  // not the last slice to finish
    __threadfence();
    const float4 *base = sp.partials + static_cast<size_t>(tile) * sp.split * 1024;
#pragma unroll 1
    for (int sl = 0; sl < sp.split; ++sl) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int r = j >> 2, q = j & 3;
            const float4 v = __ldcg(base + static_cast<size_t>(sl) * 1024 + j * 32 + lane);
            if (sl == 0) {
                acc[r][2 * q] = make_float2(v.x, v.y);
                acc[r][2 * q + 1] = make_float2(v.z, v.w);
            } else {
                acc[r][2 * q].x += v.x;
                acc[r][2 * q].y += v.y;
                acc[r][2 * q + 1].x += v.z;
                acc[r][2 * q + 1].y += v.w;
            }
        }
    }
    if (lane == 0) sp.counters[tile] = 0u;  // ready for the next launch on this stream
    epilogue(p, Cb, m0 + tr, n0 + 4 * tc, acc);
}

cudaError_t launch_small_splitk(const SimtProblem &p, cudaStream_t stream, const char **detail) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) {
        *detail = "cudaGetDevice failed";
        return err;
    }
    SmallParams sp;
    KParams &kp = sp.k;
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
    kp.tiles_m = (p.M + 63) / 64;
    kp.tiles_n = (p.N + 63) / 64;
    kp.group_m = 8;
    kp.a_vec4 = operand_vec4(p.A, p.lda, p.strideA, p.batch);
    kp.b_vec4 = operand_vec4(p.B, p.ldb, p.strideB, p.batch);
    kp.c_vec4 = operand_vec4(p.C, p.ldc, p.strideC, p.batch);
    kp.bias = p.bias;
    kp.act = p.act;
    const long long tiles = static_cast<long long>(kp.tiles_m) * kp.tiles_n * p.batch;
    if (tiles > 0x7fffffffLL) {
        *detail = "too many output tiles for the split-K grid";
        return cudaErrorInvalidValue;
    }
    // Slices: enough one-warp CTAs for about four per SM, at most 16 and at most one per
    // 32-wide k-tile; then no empty slice.
    const long long KT = (p.K + BK - 1) / BK;
    const int sms = std::max(1, device_sms(dev));
    long long split = (4LL * sms + tiles - 1) / tiles;
    split = std::min<long long>(std::min<long long>(split, 16), std::max<long long>(KT, 1));
    if (split < 1) split = 1;
    const long long per = (KT + split - 1) / split;
    split = per > 0 ? (KT + per - 1) / per : 1;
    if (split < 1) split = 1;
    sp.split = static_cast<int>(split);
    sp.kt_per_slice = static_cast<int>(per > 0 ? per : 1);
    sp.partials = nullptr;
    sp.counters = nullptr;
    if (split > 1) {
        // The counts live in their own allocation: zeroed whenever it is (re)allocated, and
        // left at zero by every launch (the last slice of each tile resets its count), so any
        // later launch on this stream, of any tile count that fits, starts from zeros.
        float *cnt = nullptr, *ws = nullptr;
        bool fresh = false;
        const size_t count_bytes = static_cast<size_t>(tiles) * sizeof(unsigned int);
        err = pack_workspace(dev, stream, kSlotSplitKCount, count_bytes, &cnt, &fresh);
        if (err == cudaSuccess && fresh) err = cudaMemsetAsync(cnt, 0, count_bytes, stream);
        if (err == cudaSuccess)
            err = pack_workspace(dev, stream, kSlotSplitK,
                                 static_cast<size_t>(tiles) * split * 1024 * sizeof(float4), &ws);
        if (err != cudaSuccess) {
            *detail = "split-K workspace allocation failed";
            return err;
        }
        sp.counters = reinterpret_cast<unsigned int *>(cnt);
        sp.partials = reinterpret_cast<float4 *>(ws);
    }
    small_splitk_kernel<<<dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(split)), 32, 0,
                          stream>>>(sp);
    err = cudaGetLastError();
    if (err != cudaSuccess) *detail = "kernel launch failed";
    return err;
}

cudaError_t launch_packed(int inner, const SimtProblem &p, cudaStream_t stream,
                          const char **detail) {
    const bool packA = !operand_vec4(p.A, p.lda, p.strideA, p.batch);
    const bool packB = !operand_vec4(p.B, p.ldb, p.strideB, p.batch);
    const long long ldA = (static_cast<long long>(p.K) + 3) / 4 * 4;
    const long long ldB = (static_cast<long long>(p.N) + 3) / 4 * 4;
    const long long elemsA = packA ? static_cast<long long>(p.M) * ldA : 0;
    const long long elemsB = packB ? static_cast<long long>(p.K) * ldB : 0;
    SimtProblem q = p;
    if (packA || packB) {
        int dev = 0;
        cudaError_t err = cudaGetDevice(&dev);
        if (err != cudaSuccess) {
            *detail = "cudaGetDevice failed";
            return err;
        }
        float *ws = nullptr;
        err = pack_workspace(dev, stream, kSlotRealigned,
                             static_cast<size_t>(elemsA + elemsB) * p.batch * 4, &ws);
        if (err != cudaSuccess) {
            *detail = "repacking workspace allocation failed";
            return err;
        }
        if (packA) {
            pack_rows_kernel<<<rows_grid(static_cast<long long>(p.M) * p.batch, p.K), 256, 0,
                               stream>>>(p.A, p.lda, p.strideA, ws, ldA, elemsA, p.M, p.K,
                                         p.batch);
            q.A = ws;
            q.lda = ldA;
            q.strideA = p.batch > 1 ? elemsA : 0;
        }
        if (packB) {
            float *wb = ws + elemsA * p.batch;
            pack_rows_kernel<<<rows_grid(static_cast<long long>(p.K) * p.batch, p.N), 256, 0,
                               stream>>>(p.B, p.ldb, p.strideB, wb, ldB, elemsB, p.K, p.N,
                                         p.batch);
            q.B = wb;
            q.ldb = ldB;
            q.strideB = p.batch > 1 ? elemsB : 0;
        }
        err = cudaGetLastError();
        if (err != cudaSuccess) {
            *detail = "repacking kernel launch failed";
            return err;
        }
    }
    if (!tma_ok(q)) {
        *detail = "operands not readable by TMA after repacking";
        return cudaErrorInvalidValue;
    }
    return simt_launch(inner, q, stream, detail);
}

}  // namespace

cudaError_t release_pack_workspaces() {
    std::lock_guard<std::mutex> lock(g_pack_mutex);
    cudaError_t first = cudaSuccess;
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto &w : g_pack_ws) {
        if (!w.ptr) continue;
        cudaSetDevice(w.dev);
        cudaError_t err = cudaFree(w.ptr);
        if (err != cudaSuccess && first == cudaSuccess) first = err;
    }
    cudaSetDevice(cur);
    g_pack_ws.clear();
    return first;
}

// ---- transposed operands -------------------------------------------------------------------------
namespace {

// src (rows x cols, leading dimension lds, batch stride ss) -> dst (cols x rows, ldd, sd)
// through a 32 x 33 shared tile: reads along a src row and writes along a dst row are both
// coalesced.
__global__ void __launch_bounds__(256)
    transpose_kernel(const float *__restrict__ src, long long lds, long long ss,
                     float *__restrict__ dst, long long ldd, long long sd, int rows, int cols) {
    __shared__ float tile[32][33];
    const int b = blockIdx.z;
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    const float *sb = src + b * ss;
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
        const int r = r0 + ty + j, c = c0 + tx;
        tile[ty + j][tx] = (r < rows && c < cols) ? sb[static_cast<long long>(r) * lds + c] : 0.0f;
    }
    __syncthreads();
    float *db = dst + b * sd;
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
        const int c = c0 + ty + j, r = r0 + tx;  // dst row c, column r
        if (c < cols && r < rows) db[static_cast<long long>(c) * ldd + r] = tile[tx][ty + j];
    }
}

}  // namespace

cudaError_t simt_untranspose(const SimtProblem &p, cudaStream_t stream, SimtProblem *q,
                             const char **detail) {
    *q = p;
    q->transA = false;
    q->transB = false;
    if (!p.transA && !p.transB) return cudaSuccess;
    // A broadcast operand (batch stride 0) is transposed once and stays broadcast.
    const int nbA = (p.batch > 1 && p.strideA == 0) ? 1 : p.batch;
    const int nbB = (p.batch > 1 && p.strideB == 0) ? 1 : p.batch;
    const long long ldA = (static_cast<long long>(p.K) + 3) / 4 * 4;  // new A: M x K
    const long long ldB = (static_cast<long long>(p.N) + 3) / 4 * 4;  // new B: K x N
    const long long elemsA = p.transA ? static_cast<long long>(p.M) * ldA : 0;
    const long long elemsB = p.transB ? static_cast<long long>(p.K) * ldB : 0;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) {
        *detail = "cudaGetDevice failed";
        return err;
    }
    float *ws = nullptr;
    err = pack_workspace(dev, stream, kSlotTransposed,
                         static_cast<size_t>(elemsA * nbA + elemsB * nbB) * 4, &ws);
    if (err != cudaSuccess) {
        *detail = "transpose workspace allocation failed";
        return err;
    }
    if (p.transA) {  // A stored K x M -> M x K
        dim3 grid((p.M + 31) / 32, (p.K + 31) / 32, nbA);
        transpose_kernel<<<grid, 256, 0, stream>>>(p.A, p.lda, p.strideA, ws, ldA, elemsA, p.K,
                                                   p.M);
        q->A = ws;
        q->lda = ldA;
        q->strideA = nbA > 1 ? elemsA : 0;
    }
    if (p.transB) {  // B stored N x K -> K x N
        float *wb = ws + elemsA * nbA;
        dim3 grid((p.K + 31) / 32, (p.N + 31) / 32, nbB);
        transpose_kernel<<<grid, 256, 0, stream>>>(p.B, p.ldb, p.strideB, wb, ldB, elemsB, p.N,
                                                   p.K);
        q->B = wb;
        q->ldb = ldB;
        q->strideB = nbB > 1 ? elemsB : 0;
    }
    err = cudaGetLastError();
    if (err != cudaSuccess) *detail = "transpose kernel launch failed";
    return err;
}

}  // namespace sg
