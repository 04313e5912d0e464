// tf32x3_gemm.cu: C = alpha * (A . B) + beta * C on the tcgen05 tensor cores, fp32 emulated by
// three TF32 products (the published "3xTF32" split; the pages mention tensor cores only in
// passing, as the way past the SIMT ladder, "GEMM scrapbook", closing remarks).
//
// Split. Every operand value x becomes big = tf32_rna(x) and small = tf32_rna(x - big); big
// has the low 13 mantissa bits clear, x - big is exact in fp32, and big.big + big.small +
// small.big misses only small.small (about 2^-22 relative) and the rounding of small. A
// pre-pass writes A's parts row-major (K contiguous) and B's parts transposed (N x K, K
// contiguous), so both MMA operands are K-major in shared memory. Non-finite values keep
// big = x and small = 0, so Inf and NaN propagate as in fp32; finite values whose rounding
// would overflow (within half a TF32 step of FLT_MAX) are truncated instead.
//
// GEMM. A persistent grid (one CTA per SM) walks the 128 x BN output tiles in grouped-raster
// order, tile t, t + grid, ...; 6 warps per CTA:
//   warp 0, lane 0: TMA producer, four boxes per 32-wide k-block (A big/small 128 x 32,
//                   B big/small BN x 32, 128-byte swizzle) into a STAGES-deep ring that runs
//                   on from one tile into the next;
//   warp 1:         allocates two sets of ACCS x BN TMEM columns (one per tile in flight);
//                   lane 0 issues the MMAs: per k-block 4 k-steps x (small_A.big_B,
//                   big_A.small_B, big_A.big_B), each tcgen05.mma.cta_group::1.kind::tf32
//                   M=128, N=BN, K=8, accumulating in TMEM (fp32); k-block kb goes to
//                   accumulator kb % ACCS of the tile's set; tcgen05.commit frees each stage,
//                   and a commit per tile marks its set ready;
//   warps 2..5:     epilogue: tcgen05.ld (32 lanes x 32 columns per load) of the TMEM rows the
//                   warp may access, the ACCS accumulators summed in fp32 in a fixed order,
//                   alpha * acc + beta * C (C unread when beta == 0), stores; after its last
//                   load of a tile each warp hands the set back, so tile j's epilogue runs
//                   while the MMAs of tile j + 1 fill the other set.
// Why several accumulators: the tensor core's fp32 accumulation loses more than round-to-
// nearest as the running sum grows (measured: normalised error 7.2e-6 at K = 16384 with one
// accumulator). The error grows like n^1.5 for n terms per accumulator, so ACCS accumulators
// over interleaved k-blocks cut it by about sqrt(ACCS).
// Every wait is bounded; a wait that expires raises the fault word, the role stops, the TMA
// producer waits (bounded) for the copies it issued to land, and the CTA still meets at the
// final barrier and frees its TMEM.
//
// Single-product mode (PRODUCTS = 1, the "1xTF32" fast path): the pre-pass writes only the big
// parts (tf32_rna of each value) and the kernel issues big_A.big_B alone, with twice the
// stages in the same shared memory. Each product is then off by at most (2u + u^2)|a b|,
// u = 2^-11, so the result carries TF32 rather than fp32 accuracy.
#include "epilogue.cuh"
#include "ptx.cuh"
#include "raster.cuh"
#include "tf32x3_gemm.cuh"

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

namespace sg {
namespace {

constexpr int BM = 128;
constexpr int BK = 32;  // fp32 values per 128-byte swizzled row

// ---- split pre-pass -------------------------------------------------------------------------

__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// x = big + small. A finite x within half a TF32 step of FLT_MAX rounds up past the largest
// exponent; for those, big keeps x's top bits (truncation) so that big stays finite and
// small = x - big is exact. Non-finite x: big = x, small = 0.
__device__ __forceinline__ void split_value(float x, float &big, float &small) {
    big = tf32_rna(x);
    if (isfinite(big)) {
        small = tf32_rna(x - big);
    } else if (isfinite(x)) {
        big = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
        small = tf32_rna(x - big);
    } else {
        small = 0.0f;
    }
}

// One operand's share of the split pre-pass. A rows job keeps the orientation: src (rows x
// cols, leading dimension ld, batch stride stride) -> big, small (rows x ldo each, batch
// stride so; ldo and so multiples of 4, outputs 16-byte aligned). A transposing job writes
// src (rows = K x cols = N) as N x K (K contiguous). Both operands' jobs run in one launch:
// CTAs [0, j0.blocks) take the first job, the rest the second.
struct SplitJob {
    const float *src;
    long long ld, stride;
    float *big, *small;
    long long ldo, so;
    int rows, cols, batch;
    int transpose;  // 0: rows job, 1: transposing job
    int vec;        // 16-byte source reads allowed
    int gx, gy;     // the job's CTA grid: rows job gx x gy; transposing job gx x gy x batch
    long long tiles;   // transposing job: 32 x 32 tiles in all (the CTAs loop over them)
    long long blocks;  // CTAs of this job
};

// Rows job: rows over the grid's y dimension, columns over threads, float4 access when the
// source allows.
template <bool SMALL>
__device__ __forceinline__ void split_rows(const SplitJob &j, long long bid) {
    const int bx = static_cast<int>(bid % j.gx);
    const long long by = bid / j.gx;
    const long long nrows = static_cast<long long>(j.rows) * j.batch;
    const int stride = j.gx * blockDim.x;
    for (long long gr = by; gr < nrows; gr += j.gy) {
        const long long b = gr / j.rows, r = gr - b * j.rows;
        const float *src = j.src + b * j.stride + r * j.ld;
        float *hi = j.big + b * j.so + r * j.ldo;
        float *lo = j.small + b * j.so + r * j.ldo;
        const int c4 = j.vec ? (j.cols & ~3) : 0;
        for (int c = 4 * (bx * blockDim.x + threadIdx.x); c < c4; c += 4 * stride) {
            const float4 x = __ldcs(reinterpret_cast<const float4 *>(src + c));
            float4 h, l;
            split_value(x.x, h.x, l.x);
            split_value(x.y, h.y, l.y);
            split_value(x.z, h.z, l.z);
            split_value(x.w, h.w, l.w);
            *reinterpret_cast<float4 *>(hi + c) = h;
            if (SMALL) *reinterpret_cast<float4 *>(lo + c) = l;
        }
        for (int c = c4 + bx * blockDim.x + threadIdx.x; c < j.cols; c += stride) {
            float h, l;
            split_value(src[c], h, l);
            hi[c] = h;
            if (SMALL) lo[c] = l;
        }
    }
}

// Transposing job: a 32 x 32 tile goes through shared memory; 256 threads each read one
// float4 along n (when the source allows) and write one float4 along k of each output, so
// both sides move 16 bytes per thread.
template <bool SMALL>
__device__ __forceinline__ void split_transpose_tile(const SplitJob &j, long long bid,
                                                     float (&tile)[32][33]) {
    const int K = j.rows, N = j.cols;
    const int n0 = static_cast<int>(bid % j.gx) * 32;
    const long long rest = bid / j.gx;
    const int k0 = static_cast<int>(rest % j.gy) * 32;
    const long long b = rest / j.gy;
    const int t = threadIdx.x;
    const float *Bb = j.src + b * j.stride;
    {
        const int kr = t >> 3, nc = (t & 7) * 4;  // row k0 + kr, columns n0 + nc .. + 3
        const int k = k0 + kr, n = n0 + nc;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (k < K) {
            const float *src = Bb + static_cast<long long>(k) * j.ld + n;
            if (j.vec && n + 3 < N) {
                v = __ldcs(reinterpret_cast<const float4 *>(src));
            } else {
                if (n < N) v.x = src[0];
                if (n + 1 < N) v.y = src[1];
                if (n + 2 < N) v.z = src[2];
                if (n + 3 < N) v.w = src[3];
            }
        }
        tile[kr][nc] = v.x;
        tile[kr][nc + 1] = v.y;
        tile[kr][nc + 2] = v.z;
        tile[kr][nc + 3] = v.w;
    }
    __syncthreads();
    {
        const int nr = t >> 3, kc = (t & 7) * 4;  // output row n0 + nr, k0 + kc .. + 3
        const int n = n0 + nr, k = k0 + kc;
        if (n < N) {
            float4 h, l;
            split_value(tile[kc][nr], h.x, l.x);
            split_value(tile[kc + 1][nr], h.y, l.y);
            split_value(tile[kc + 2][nr], h.z, l.z);
            split_value(tile[kc + 3][nr], h.w, l.w);
            float *ob = j.big + b * j.so + static_cast<long long>(n) * j.ldo + k;
            float *os = j.small + b * j.so + static_cast<long long>(n) * j.ldo + k;
            if (k + 3 < K) {
                *reinterpret_cast<float4 *>(ob) = h;
                if (SMALL) *reinterpret_cast<float4 *>(os) = l;
            } else {
                const float hv[4] = {h.x, h.y, h.z, h.w}, lv[4] = {l.x, l.y, l.z, l.w};
                for (int e = 0; e < 4 && k + e < K; ++e) {
                    ob[e] = hv[e];
                    if (SMALL) os[e] = lv[e];
                }
            }
        }
    }
}

// The transposing job's CTAs walk its tiles with a stride of the job's CTA count.
template <bool SMALL>
__device__ __forceinline__ void split_transpose(const SplitJob &j, long long bid,
                                                float (&tile)[32][33]) {
    for (long long t = bid; t < j.tiles; t += j.blocks) {
        split_transpose_tile<SMALL>(j, t, tile);
        __syncthreads();  // the tile buffer is reused by the next tile
    }
}

// Both operands' split in one launch. The GEMM that follows is launched as a programmatic
// dependent: every CTA here lets it start its prologue at once, and it waits for this grid's
// completion (griddepcontrol.wait) before it reads a split operand.
template <bool SMALL>
__global__ void __launch_bounds__(256) split_operands_kernel(const SplitJob j0, const SplitJob j1) {
    __shared__ float tile[32][33];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    long long bid = blockIdx.x;
    const bool first = bid < j0.blocks;
    const SplitJob &j = first ? j0 : j1;
    if (!first) bid -= j0.blocks;
    if (j.transpose)
        split_transpose<SMALL>(j, bid, tile);
    else
        split_rows<SMALL>(j, bid);
}

// ---- tcgen05 wrappers ---------------------------------------------------------------------------

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 bytes
// apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);   // start address
    d |= static_cast<uint64_t>(1u) << 16;                  // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;          // stride byte offset
    d |= static_cast<uint64_t>(1u) << 46;                  // version
    d |= static_cast<uint64_t>(2u) << 61;                  // swizzle: 128 bytes
    return d;
}

// Instruction descriptor: D fp32, A and B tf32, both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_tf32(int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(BM >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t gets lane (base lane + t), 32 values.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

struct TParams {
    int M, N, K;
    float alpha, beta;
    float *C;
    long long ldc, sC;
    int batch;
    int tiles_m, tiles_n, group_m;
    int total_tiles;    // tiles_m * tiles_n * batch
    int c_vec4;
    const float *bias;  // fused epilogue (nullptr: none)
    int act;            // fused epilogue activation (0: none)
};

__host__ __device__ constexpr uint32_t pow2_at_least(uint32_t v) {
    uint32_t r = 32;
    while (r < v) r <<= 1;
    return r;
}

template <int BN, int STAGES, int ACCS, int PRODUCTS>
__global__ void __launch_bounds__(192, 1)
    tf32x3_gemm_kernel(const __grid_constant__ CUtensorMap mapAhi,
                       const __grid_constant__ CUtensorMap mapAlo,
                       const __grid_constant__ CUtensorMap mapBhi,
                       const __grid_constant__ CUtensorMap mapBlo, const TParams p) {
    constexpr uint32_t A_BYTES = BM * BK * 4;  // 16 KiB per part
    constexpr uint32_t B_BYTES = BN * BK * 4;
    static_assert(PRODUCTS == 3 || PRODUCTS == 1, "3xTF32 or a single TF32 product");
    constexpr uint32_t PARTS = PRODUCTS == 3 ? 2 : 1;  // big (and small) of each operand
    constexpr uint32_t STAGE_BYTES = PARTS * (A_BYTES + B_BYTES);
    constexpr uint32_t IDESC = idesc_tf32(BN);
    constexpr uint32_t SET_COLS = BN * ACCS;                   // one tile's accumulators
    constexpr uint32_t TMEM_COLS = pow2_at_least(2 * SET_COLS);  // two tiles in flight
    constexpr uint32_t SET_STRIDE = TMEM_COLS / 2;
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
    static_assert(BN % 32 == 0, "the epilogue reads 32-column slices");
    static_assert(TMEM_COLS <= 512, "two accumulator sets must fit in TMEM");
    constexpr int EPI_WARPS = 4;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *set_full = empty + STAGES;  // [2]: a tile's accumulators are complete
    uint64_t *set_free = set_full + 2;    // [2]: the epilogue has read them
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(set_free + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = (p.K + BK - 1) / BK;
    const int tiles_per_batch = p.tiles_m * p.tiles_n;

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&mapAhi);
        tma_prefetch_desc(&mapAlo);
        tma_prefetch_desc(&mapBhi);
        tma_prefetch_desc(&mapBlo);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&set_full[j], 1);
            mbar_init(&set_free[j], EPI_WARPS);
        }
        mbar_init_fence();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent of the split pass: the prologue above overlapped its
    // tail; the split operands are read only after its grid has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // Output tile t of the persistent walk: batch entry b, origin (m0, n0).
    auto tile_origin = [&](int t, int &b, int &m0, int &n0) {
        b = t / tiles_per_batch;
        int tm, tn;  // grouped raster: concurrently running tiles share A and B panels in L2
        tile_coords(t - b * tiles_per_batch, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
        m0 = tm * BM;
        n0 = tn * BN;
    };

    if (warp == 0 && lane == 0) {
        // ---- TMA producer ----
        int it = 0;  // ring position over every k-block of every tile
        bool ok = true;
        for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
            int b, m0, n0;
            tile_origin(t, b, m0, n0);
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int s = it % STAGES;
                if (it >= STAGES && !mbar_wait(&empty[s], ((it / STAGES) - 1) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t *st = smem + s * STAGE_BYTES;
                mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                tma_load_3d(st, &mapAhi, &full[s], kb * BK, m0, b);
                tma_load_3d(st + PARTS * A_BYTES, &mapBhi, &full[s], kb * BK, n0, b);
                if (PRODUCTS == 3) {
                    tma_load_3d(st + A_BYTES, &mapAlo, &full[s], kb * BK, m0, b);
                    tma_load_3d(st + 2 * A_BYTES + B_BYTES, &mapBlo, &full[s], kb * BK, n0, b);
                }
            }
        }
        // The CTA's shared memory must outlive every copy: wait (bounded) for the last
        // STAGES issued to land; stages the MMAs already consumed complete at once.
        for (int j = it > STAGES ? it - STAGES : 0; j < it; ++j)
            if (!mbar_wait(&full[j % STAGES], (j / STAGES) & 1)) break;
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----
        int it = 0, j = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x, ++j) {
            const int set = j & 1;
            if (j >= 2 && !mbar_wait(&set_free[set], ((j >> 1) - 1) & 1)) break;
            tc_fence_after();
            const uint32_t dset = tmem + static_cast<uint32_t>(set) * SET_STRIDE;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int s = it % STAGES;
                if (!mbar_wait(&full[s], (it / STAGES) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t st = smem_addr(smem + s * STAGE_BYTES);
                const uint32_t a_hi = st, a_lo = st + A_BYTES;
                const uint32_t b_hi = st + PARTS * A_BYTES, b_lo = b_hi + B_BYTES;
                const uint32_t d = dset + static_cast<uint32_t>((kb % ACCS) * BN);
#pragma unroll
                for (int kk = 0; kk < BK / 8; ++kk) {
                    const uint32_t off = kk * 32;  // 8 tf32 values along k
                    const uint32_t acc0 = (kb >= ACCS || kk > 0) ? 1u : 0u;  // first: overwrite
                    if (PRODUCTS == 3) {
                        mma_tf32(d, smem_desc_sw128(a_lo + off), smem_desc_sw128(b_hi + off), IDESC, acc0);
                        mma_tf32(d, smem_desc_sw128(a_hi + off), smem_desc_sw128(b_lo + off), IDESC, 1u);
                        mma_tf32(d, smem_desc_sw128(a_hi + off), smem_desc_sw128(b_hi + off), IDESC, 1u);
                    } else {
                        mma_tf32(d, smem_desc_sw128(a_hi + off), smem_desc_sw128(b_hi + off), IDESC, acc0);
                    }
                }
                mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
            }
            if (ok) mma_commit(&set_full[set]);  // arrives when this tile's MMAs are complete
        }
    } else if (warp >= 2) {
        // ---- epilogue: TMEM -> registers -> C ----
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int used = KB < ACCS ? KB : ACCS;  // accumulators that received k-blocks
        const float alpha = p.alpha, beta = p.beta;
        int j = 0;
        for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++j) {
            const int set = j & 1;
            if (!mbar_wait(&set_full[set], (j >> 1) & 1)) break;
            tc_fence_after();
            int b, m0, n0;
            tile_origin(t, b, m0, n0);
            const uint32_t tset = tmem + lane_base + static_cast<uint32_t>(set) * SET_STRIDE;
            const int row = m0 + quarter * 32 + lane;
            float *crow = p.C + static_cast<long long>(b) * p.sC + static_cast<long long>(row) * p.ldc;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                float v[32];
                tmem_ld_32x32b_x32(tset + c0, v);
                for (int a = 1; a < used; ++a) {
                    float w[32];
                    tmem_ld_32x32b_x32(tset + static_cast<uint32_t>(a * BN + c0), w);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] += w[i];
                }
                if (c0 + 32 >= BN) {
                    // Last slice read: hand the set back to the MMA issuer.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&set_free[set]);
                }
                if (row >= p.M || KB == 0) continue;
                const int col0 = n0 + c0;
                const bool vec = p.c_vec4 && col0 + 31 < p.N;
                // beta != 0: the slice's 32 C values are loaded before any store (a store may
                // alias a later load as far as the compiler knows).
                float cv[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) cv[jj] = 0.0f;
                if (beta != 0.0f) {
                    if (vec) {
#pragma unroll
                        for (int jj = 0; jj < 32; jj += 4) {
                            const float4 c = *reinterpret_cast<const float4 *>(crow + col0 + jj);
                            cv[jj] = c.x;
                            cv[jj + 1] = c.y;
                            cv[jj + 2] = c.z;
                            cv[jj + 3] = c.w;
                        }
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj)
                            if (col0 + jj < p.N) cv[jj] = crow[col0 + jj];
                    }
                }
                const bool fused = p.bias != nullptr || p.act != kActNone;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                    v[jj] = fused ? epilogue_apply(v[jj], alpha, beta, p.bias, col0 + jj, p.act, cv[jj])
                                  : (beta != 0.0f ? fmaf(alpha, v[jj], beta * cv[jj]) : alpha * v[jj]);
                if (vec) {
#pragma unroll
                    for (int jj = 0; jj < 32; jj += 4)
                        *reinterpret_cast<float4 *>(crow + col0 + jj) =
                            make_float4(v[jj], v[jj + 1], v[jj + 2], v[jj + 3]);
                } else {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        if (col0 + jj < p.N) crow[col0 + jj] = v[jj];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();  // every role is done with the ring and the accumulators
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

// ---- host side ------------------------------------------------------------------------------

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

// A K-major split operand: `rows` x K values, row stride ldk, `batch` copies `stride` apart;
// boxes of box_rows x 32 with the 128-byte swizzle.
bool make_split_map(CUtensorMap *map, const float *base, long long rows, long long K,
                    long long ldk, long long stride, int batch, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldk * 4), static_cast<cuuint64_t>(stride * 4)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct SplitWorkspace {
    int dev;
    cudaStream_t stream;
    void *ptr;
    size_t bytes;
};
std::mutex g_split_mutex;
std::vector<SplitWorkspace> g_split_ws;

cudaError_t split_workspace(int dev, cudaStream_t stream, size_t bytes, float **out) {
    std::lock_guard<std::mutex> lock(g_split_mutex);
    SplitWorkspace *e = nullptr;
    for (auto &w : g_split_ws)
        if (w.dev == dev && w.stream == stream) e = &w;
    if (e && e->bytes < bytes) {
        cudaError_t err = cudaFree(e->ptr);
        e->ptr = nullptr;
        e->bytes = 0;
        if (err != cudaSuccess) return err;
    }
    if (!e) {
        g_split_ws.push_back({dev, stream, nullptr, 0});
        e = &g_split_ws.back();
    }
    if (!e->ptr) {
        cudaError_t err = cudaMalloc(&e->ptr, bytes);
        if (err != cudaSuccess) {
            e->ptr = nullptr;
            return err;
        }
        e->bytes = bytes;
    }
    *out = static_cast<float *>(e->ptr);
    return cudaSuccess;
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

constexpr int kMaxDevices = 64;

// Multiprocessors of device `dev` (queried once), or 0 if the query fails.
int sm_count(int dev) {
    static std::once_flag once[kMaxDevices];
    static int count[kMaxDevices];
    std::call_once(once[dev], [&] {
        if (cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            count[dev] = 0;
    });
    return count[dev];
}

SplitJob make_job(const float *src, long long ld, long long stride, float *big, float *small,
                  long long ldo, long long so, int rows, int cols, int batch, bool transpose,
                  bool vec) {
    SplitJob j;
    j.src = src;
    j.ld = ld;
    j.stride = stride;
    j.big = big;
    j.small = small;
    j.ldo = ldo;
    j.so = so;
    j.rows = rows;
    j.cols = cols;
    j.batch = batch;
    j.transpose = transpose ? 1 : 0;
    j.vec = vec ? 1 : 0;
    // About 4,096 CTAs per job, each looping over several rows or tiles: CTAs of a single
    // 4 KiB row chunk or tile spent a large share of their time starting up.
    if (transpose) {  // 32 x 32 tiles of the rows x cols source, per batch entry
        j.gx = (cols + 31) / 32;
        j.gy = (rows + 31) / 32;
        j.tiles = static_cast<long long>(j.gx) * j.gy * batch;
        j.blocks = std::min<long long>(j.tiles, 4096);
    } else {  // up to 8 CTAs of 1024 columns across a row, rows (of every batch entry) down
        const long long nrows = static_cast<long long>(rows) * batch;
        j.gx = static_cast<int>(std::max<long long>(1, std::min<long long>((cols + 1023) / 1024, 8)));
        j.gy = static_cast<int>(std::max<long long>(1, std::min<long long>(nrows, 4096 / j.gx)));
        j.tiles = 0;
        j.blocks = static_cast<long long>(j.gx) * j.gy;
    }
    return j;
}

template <int BN, int STAGES, int ACCS, int PRODUCTS>
cudaError_t launch_tf32x3(const SimtProblem &p, cudaStream_t stream, const char **detail) {
    constexpr size_t PARTS = PRODUCTS == 3 ? 2 : 1;
    constexpr size_t STAGE_BYTES = PARTS * (BM * BK * 4 + static_cast<size_t>(BN) * BK * 4);
    constexpr size_t SMEM = STAGES * STAGE_BYTES + (2 * STAGES + 4) * 8 + 16 + 1024;
    auto kernel = tf32x3_gemm_kernel<BN, STAGES, ACCS, PRODUCTS>;

    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *detail = "cudaGetDevice failed";
        return err != cudaSuccess ? err : cudaErrorInvalidDevice;
    }
    static std::once_flag once[kMaxDevices];
    static cudaError_t attr_err[kMaxDevices];
    std::call_once(once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(SMEM));
    });
    if (attr_err[dev] != cudaSuccess) {
        *detail = "cudaFuncSetAttribute(max dynamic shared memory) failed";
        return attr_err[dev];
    }
    const int sms = sm_count(dev);
    if (sms <= 0) {
        *detail = "multiprocessor count query failed";
        return cudaErrorInvalidDevice;
    }

    // Split workspace: A parts M x ldk, B parts N x ldk (ldk = K rounded up to 4 so rows
    // start 16-byte aligned for TMA), per batch entry.
    const long long ldk = (static_cast<long long>(p.K) + 3) / 4 * 4;
    const long long a_elems = static_cast<long long>(p.M) * ldk;
    const long long b_elems = static_cast<long long>(p.N) * ldk;
    const long long per_batch = static_cast<long long>(PARTS) * (a_elems + b_elems);
    float *ws = nullptr;
    err = split_workspace(dev, stream, static_cast<size_t>(per_batch) * p.batch * 4, &ws);
    if (err != cudaSuccess) {
        *detail = "3xTF32 split workspace allocation failed";
        return err;
    }
    float *a_hi = ws;
    float *a_lo = PARTS == 2 ? a_hi + a_elems * p.batch : a_hi;
    float *b_hi = a_lo + a_elems * p.batch;
    float *b_lo = PARTS == 2 ? b_hi + b_elems * p.batch : b_hi;
    constexpr bool SMALL = PARTS == 2;

    {
        const bool vecA = aligned16(p.A) && p.lda % 4 == 0 && (p.batch <= 1 || p.strideA % 4 == 0);
        const bool vecB = aligned16(p.B) && p.ldb % 4 == 0 && (p.batch <= 1 || p.strideB % 4 == 0);
        // A -> M x K (K contiguous): a rows job, or a transposing job when A is stored K x M.
        // B -> N x K (K contiguous): a transposing job, or a rows job when B is stored N x K.
        SplitJob ja = make_job(p.A, p.lda, p.strideA, a_hi, a_lo, ldk, a_elems, p.transA ? p.K : p.M,
                               p.transA ? p.M : p.K, p.batch, p.transA, vecA);
        SplitJob jb = make_job(p.B, p.ldb, p.strideB, b_hi, b_lo, ldk, b_elems, p.transB ? p.N : p.K,
                               p.transB ? p.K : p.N, p.batch, !p.transB, vecB);
        const long long blocks = ja.blocks + jb.blocks;
        if (blocks > 0x7fffffffLL) {
            *detail = "split pre-pass grid too large";
            return cudaErrorInvalidValue;
        }
        split_operands_kernel<SMALL><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(ja, jb);
        err = cudaGetLastError();
        if (err != cudaSuccess) {
            *detail = "split kernel launch failed";
            return err;
        }
    }

    CUtensorMap mAhi, mAlo, mBhi, mBlo;
    if (!make_split_map(&mAhi, a_hi, p.M, p.K, ldk, a_elems, p.batch, BM) ||
        !make_split_map(&mAlo, a_lo, p.M, p.K, ldk, a_elems, p.batch, BM) ||
        !make_split_map(&mBhi, b_hi, p.N, p.K, ldk, b_elems, p.batch, BN) ||
        !make_split_map(&mBlo, b_lo, p.N, p.K, ldk, b_elems, p.batch, BN)) {
        *detail = "cuTensorMapEncodeTiled rejected a split operand";
        return cudaErrorInvalidValue;
    }
    TParams tp;
    tp.M = p.M;
    tp.N = p.N;
    tp.K = p.K;
    tp.alpha = p.alpha;
    tp.beta = p.beta;
    tp.C = p.C;
    tp.ldc = p.ldc;
    tp.sC = p.strideC;
    tp.batch = p.batch;
    tp.tiles_m = (p.M + BM - 1) / BM;
    tp.tiles_n = (p.N + BN - 1) / BN;
    tp.group_m = 16;
    tp.c_vec4 = aligned16(p.C) && p.ldc % 4 == 0 && (p.batch <= 1 || p.strideC % 4 == 0);
    tp.bias = p.bias;
    tp.act = p.act;
    const long long tiles = static_cast<long long>(tp.tiles_m) * tp.tiles_n * p.batch;
    if (tiles > 0x7fffffffLL) {
        *detail = "too many output tiles for the tensor-core grid";
        return cudaErrorInvalidValue;
    }
    tp.total_tiles = static_cast<int>(tiles);
    const int grid = static_cast<int>(std::min<long long>(tiles, sms));  // one CTA per SM
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, kernel, mAhi, mAlo, mBhi, mBlo, tp);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) *detail = "3xTF32 kernel launch failed";
    return err;
}

// Tile width of the tensor paths. The persistent grid runs ceil(tiles / SMs) rounds of tiles;
// a round costs the MMA time of one tile, proportional to BN, divided by the width's
// efficiency (narrower tiles read more shared memory per MMA; measured on a GB300 at
// 16384 x 14336 x 4096: 192 columns run at 0.953 of the rate of 256, 224 interpolated at
// 0.975). The single-product path takes the width in {256, 224, 192} with the lowest
// rounds x BN / efficiency (4096 x 4096: 608 tiles of 224 = 4 rounds, 627 TFLOP/s, against
// 548 for 4 rounds of 256 and 550 for 5 rounds of 192; 16384 x 14336: 256). The 3xTF32
// path keeps BN = 128: its two accumulators per tile (for accuracy) times two tiles in
// flight fill the 512 TMEM columns. SGEMM_TF32_TILE_N=192|224|256 forces the width.
int tf32_tile_n(const SimtProblem &p, int sms) {
    static const int forced = [] {
        const char *env = std::getenv("SGEMM_TF32_TILE_N");
        if (!env) return 0;
        const int v = std::atoi(env);
        return v == 192 || v == 224 || v == 256 ? v : 0;
    }();
    if (forced) return forced;
    const long long tm = (p.M + BM - 1) / BM;
    constexpr int widths[3] = {256, 224, 192};
    constexpr int efficiency_milli[3] = {1000, 975, 953};
    int best = 256;
    long long best_cost = -1;
    for (int w = 0; w < 3; ++w) {
        const int bn = widths[w];
        const long long tiles = tm * ((p.N + bn - 1) / bn) * p.batch;
        const long long cost = (tiles + sms - 1) / sms * bn * 1000 / efficiency_milli[w];
        if (best_cost < 0 || cost < best_cost) {
            best = bn;
            best_cost = cost;
        }
    }
    return best;
}

}  // namespace

bool tf32x3_supports(const SimtProblem &p) { return p.batch >= 1; }

cudaError_t tf32x3_launch(const SimtProblem &p, cudaStream_t stream, const char **detail) {
    return launch_tf32x3<128, 3, 2, 3>(p, stream, detail);
}

cudaError_t tf32_launch(const SimtProblem &p, cudaStream_t stream, const char **detail) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *detail = "cudaGetDevice failed";
        return cudaErrorInvalidDevice;
    }
    switch (tf32_tile_n(p, std::max(1, sm_count(dev)))) {
        case 192: return launch_tf32x3<192, 5, 1, 1>(p, stream, detail);
        case 224: return launch_tf32x3<224, 5, 1, 1>(p, stream, detail);
        default: return launch_tf32x3<256, 4, 1, 1>(p, stream, detail);
    }
}

cudaError_t tf32x3_release_workspaces() {
    std::lock_guard<std::mutex> lock(g_split_mutex);
    cudaError_t first = cudaSuccess;
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto &w : g_split_ws) {
        if (!w.ptr) continue;
        cudaSetDevice(w.dev);
        cudaError_t err = cudaFree(w.ptr);
        if (err != cudaSuccess && first == cudaSuccess) first = err;
    }
    cudaSetDevice(cur);
    g_split_ws.clear();
    return first;
}


}  // namespace sg
