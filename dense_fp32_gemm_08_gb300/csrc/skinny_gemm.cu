// skinny_gemm.cu: bandwidth kernels for C = alpha * (A . B) + beta * C when one output
// dimension is at most 8. Such products do 2 FLOP per element of the large operand, far
// below the GB300's FP32 ridge of about 12 FLOP/B, so they are bound by streaming that
// operand from HBM once; the tile kernels would leave most SMs idle.
//
// * N <= 8 ("tall"): the large operand is A (M x K). One warp per row of A: each lane reads
//   float4 (or scalar) chunks of the row, multiplies them by the matching rows of B (K x N,
//   small and L1/L2-resident), and keeps N partial sums; a shuffle tree in fixed lane order
//   reduces them. Every row is independent; M rows give M warps of work.
// * M <= 8 ("wide"): the large operand is B (K x N). A CTA of 32 warps (16 when M > 2, 8 when
//   M > 4) owns 128 columns of C; its 8-CTA cluster splits K into 8 ranges, and within a CTA
//   warp w takes k = w, w + W, ... of its range (W warps), so every warp streams whole
//   512-byte row segments of B. Partial sums are
//   reduced over the warps through shared memory and over the cluster through distributed
//   shared memory, both in a fixed order; the cluster's CTA 0 applies alpha / beta. No
//   workspace is used, and results are deterministic.
#include <cooperative_groups.h>

#include "epilogue.cuh"
#include "ptx.cuh"
#include "skinny_gemm.cuh"

namespace cg = cooperative_groups;

namespace sg {
namespace {

// ---- tall: N <= 8 ------------------------------------------------------------------------------

template <int NN, bool VEC>
__global__ void __launch_bounds__(256) skinny_tall_kernel(SkinnyProblem p) {
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const long long gwarp = static_cast<long long>(blockIdx.x) * warps + (threadIdx.x >> 5);
    const long long nwarps = static_cast<long long>(gridDim.x) * warps;
    const long long rows = static_cast<long long>(p.M) * p.batch;
    for (long long gr = gwarp; gr < rows; gr += nwarps) {
        const long long b = gr / p.M, row = gr - b * p.M;
        const float *a = p.A + b * p.strideA + row * p.lda;
        const float *B = p.B + b * p.strideB;
        float acc[NN];
#pragma unroll
        for (int n = 0; n < NN; ++n) acc[n] = 0.0f;
        int k = 0;
        if (VEC) {
            // 4 k-values per lane per step, 128 per warp, unrolled for loads in flight; each
            // lane adds its own k-values in ascending order. With N == 1 and B a packed,
            // aligned vector, B's four values come in one float4 as well.
            const int kv = p.K & ~127;
            const bool bvec = NN == 1 && p.ldb == 1 &&
                              (reinterpret_cast<uintptr_t>(B) & 15u) == 0;
            if (bvec) {
#pragma unroll 4
                for (int k0 = 0; k0 < kv; k0 += 128) {
                    const int kk = k0 + 4 * lane;
                    const float4 av = __ldcs(reinterpret_cast<const float4 *>(a + kk));
                    const float4 bv = __ldg(reinterpret_cast<const float4 *>(B + kk));
                    acc[0] = fmaf(av.x, bv.x, acc[0]);
                    acc[0] = fmaf(av.y, bv.y, acc[0]);
                    acc[0] = fmaf(av.z, bv.z, acc[0]);
                    acc[0] = fmaf(av.w, bv.w, acc[0]);
                }
            } else {
#pragma unroll 4
                for (int k0 = 0; k0 < kv; k0 += 128) {
                    const int kk = k0 + 4 * lane;
                    const float4 av = __ldcs(reinterpret_cast<const float4 *>(a + kk));
                    const float ae[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float *brow = B + static_cast<long long>(kk + e) * p.ldb;
#pragma unroll
                        for (int n = 0; n < NN; ++n)
                            if (n < p.N) acc[n] = fmaf(ae[e], __ldg(brow + n), acc[n]);
                    }
                }
            }
            k = kv;
        }
        for (int kk = k + lane; kk < p.K; kk += 32) {
            const float av = __ldcs(a + kk);
            const float *brow = B + static_cast<long long>(kk) * p.ldb;
#pragma unroll
            for (int n = 0; n < NN; ++n)
                if (n < p.N) acc[n] = fmaf(av, __ldg(brow + n), acc[n]);
        }
#pragma unroll
        for (int n = 0; n < NN; ++n) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[n] += __shfl_xor_sync(0xffffffffu, acc[n], off);
        }
        if (lane < p.N) {
            float s = acc[0];
#pragma unroll
            for (int n = 1; n < NN; ++n)
                if (lane == n) s = acc[n];
            float *c = p.C + b * p.strideC + row * p.ldc + lane;
            *c = epilogue_value(s, p.alpha, p.beta, p.bias, lane, p.act, c);
        }
    }
}

// ---- wide: M <= 8 --------------------------------------------------------------------------------

constexpr int kWideCols = 128;   // columns of C per CTA (32 lanes x float4)
constexpr int kCluster = 8;      // CTAs per cluster, splitting K

// Warps per CTA: as many as the reduction buffer allows in static shared memory (32 for up to
// two rows, 16 up to four, 8 for eight), so that enough row segments of B are in flight to keep
// HBM busy (measured at 1 x 4096 x 4096: 32 warps 18.1 us, 16 warps 19.1 us, 8 warps 21.1 us).
template <int MM>
__host__ __device__ constexpr int wide_warps() { return MM <= 2 ? 32 : MM <= 4 ? 16 : 8; }

template <int MM, bool VEC>
__global__ void __cluster_dims__(1, kCluster, 1) __launch_bounds__(wide_warps<MM>() * 32)
    skinny_wide_kernel(SkinnyProblem p) {
    constexpr int kWideWarps = wide_warps<MM>();
    __shared__ float4 part[kWideWarps][MM][32];
    cg::cluster_group cluster = cg::this_cluster();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rank = static_cast<int>(cluster.block_rank());  // position along K
    const int b = blockIdx.z;
    const int n0 = blockIdx.x * kWideCols + 4 * lane;
    // K range of this CTA (rounded up to a multiple of 4).
    const int kper = ((p.K + kCluster - 1) / kCluster + 3) & ~3;
    const int kb = rank * kper;
    const int ke = min(p.K, kb + kper);
    const float *A = p.A + static_cast<long long>(b) * p.strideA;
    const float *B = p.B + static_cast<long long>(b) * p.strideB;

    float4 acc[MM];
#pragma unroll
    for (int m = 0; m < MM; ++m) acc[m] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const bool full = n0 + 3 < p.N;
#pragma unroll 8
    for (int k = kb + warp; k < ke; k += kWideWarps) {
        const float *brow = B + static_cast<long long>(k) * p.ldb + n0;
        float4 bv;
        if (VEC && full) {
            bv = __ldcs(reinterpret_cast<const float4 *>(brow));
        } else {
            bv.x = n0 < p.N ? __ldcs(brow) : 0.0f;
            bv.y = n0 + 1 < p.N ? __ldcs(brow + 1) : 0.0f;
            bv.z = n0 + 2 < p.N ? __ldcs(brow + 2) : 0.0f;
            bv.w = n0 + 3 < p.N ? __ldcs(brow + 3) : 0.0f;
        }
#pragma unroll
        for (int m = 0; m < MM; ++m) {
            if (m < p.M) {
                const float a = __ldg(A + static_cast<long long>(m) * p.lda + k);
                acc[m].x = fmaf(a, bv.x, acc[m].x);
                acc[m].y = fmaf(a, bv.y, acc[m].y);
                acc[m].z = fmaf(a, bv.z, acc[m].z);
                acc[m].w = fmaf(a, bv.w, acc[m].w);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MM; ++m) part[warp][m][lane] = acc[m];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int m = 0; m < MM; ++m) {
            float4 s = part[0][m][lane];
#pragma unroll
            for (int w = 1; w < kWideWarps; ++w) {
                const float4 v = part[w][m][lane];
                s.x += v.x;
                s.y += v.y;
                s.z += v.z;
                s.w += v.w;
            }
            part[0][m][lane] = s;
        }
    }
    cluster.sync();  // every CTA's partial sums are in its shared memory
    if (rank == 0 && warp == 0) {
#pragma unroll
        for (int m = 0; m < MM; ++m) {
            if (m >= p.M) continue;
            float4 s = part[0][m][lane];
            for (int r = 1; r < kCluster; ++r) {
                const float4 *remote = cluster.map_shared_rank(&part[0][m][lane], r);
                const float4 v = *remote;
                s.x += v.x;
                s.y += v.y;
                s.z += v.z;
                s.w += v.w;
            }
            float *c = p.C + static_cast<long long>(b) * p.strideC + static_cast<long long>(m) * p.ldc + n0;
            const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (n0 + e < p.N)
                    c[e] = epilogue_value(sv[e], p.alpha, p.beta, p.bias, n0 + e, p.act, c + e);
        }
    }
    cluster.sync();  // no CTA leaves while CTA 0 may still read its shared memory
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

template <int NN>
cudaError_t launch_tall(const SkinnyProblem &p, cudaStream_t stream) {
    const bool vec = aligned16(p.A) && p.lda % 4 == 0 && (p.batch <= 1 || p.strideA % 4 == 0);
    const long long rows = static_cast<long long>(p.M) * p.batch;
    long long blocks = (rows + 7) / 8;
    const long long cap = 64LL * (simt_device_sms() > 0 ? simt_device_sms() : 152);
    if (blocks > cap) blocks = cap;
    if (vec)
        skinny_tall_kernel<NN, true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    else
        skinny_tall_kernel<NN, false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int MM>
cudaError_t launch_wide(const SkinnyProblem &p, cudaStream_t stream) {
    const bool vec = aligned16(p.B) && p.ldb % 4 == 0 && (p.batch <= 1 || p.strideB % 4 == 0);
    dim3 grid((p.N + kWideCols - 1) / kWideCols, kCluster, p.batch);
    constexpr int threads = wide_warps<MM>() * 32;
    if (vec)
        skinny_wide_kernel<MM, true><<<grid, threads, 0, stream>>>(p);
    else
        skinny_wide_kernel<MM, false><<<grid, threads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool skinny_supports(int kind, const SkinnyProblem &p) {
    if (p.batch > 65535) return false;
    return kind == kSkinnyTall ? p.N <= 8 : kind == kSkinnyWide ? p.M <= 8 : false;
}

cudaError_t skinny_launch(int kind, const SkinnyProblem &p, cudaStream_t stream,
                          const char **detail) {
    cudaError_t err = cudaErrorInvalidValue;
    if (kind == kSkinnyTall && p.N <= 8) {
        err = p.N == 1 ? launch_tall<1>(p, stream)
            : p.N == 2 ? launch_tall<2>(p, stream)
            : p.N <= 4 ? launch_tall<4>(p, stream)
                       : launch_tall<8>(p, stream);
        if (err != cudaSuccess) *detail = "tall skinny kernel launch failed";
        return err;
    }
    if (kind == kSkinnyWide && p.M <= 8) {
        err = p.M == 1 ? launch_wide<1>(p, stream)
            : p.M == 2 ? launch_wide<2>(p, stream)
            : p.M <= 4 ? launch_wide<4>(p, stream)
                       : launch_wide<8>(p, stream);
        if (err != cudaSuccess) *detail = "wide skinny kernel launch failed";
        return err;
    }
    *detail = "the skinny kernel does not take this shape";
    return err;
}

}  // namespace sg
