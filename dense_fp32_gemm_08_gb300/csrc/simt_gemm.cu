// simt_gemm.cu: host side of the FP32 SIMT path: the configuration table and dispatcher, the
// state the kernel units share (tensor maps, device queries, stream-K workspaces), and the small
// kernels: operand repacking and transposition, the one-warp split-K kernel for small problems
// and the failure-path self-test. The tiled kernels themselves are templates in
// simt_kernels.cuh, instantiated by the simt_gemm_*.cu units.
#include "simt_kernels.cuh"
#include "skinny_gemm.cuh"

namespace sg {

namespace {

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

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace

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

// ---- persistent launch: workspace, grid size and the data-parallel / stream-K split ---------

namespace {
struct WorkspaceEntry {
    int dev;
    cudaStream_t stream;
    void *ptr;
    size_t bytes;
    unsigned int epoch;
};

std::mutex g_ws_mutex;
std::vector<WorkspaceEntry> g_ws;
}  // namespace


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

// Cluster size of the split-K schedule: the largest S in {8, 4, 2} whose T * S CTAs (one per
// SM) still fit on the device and that leaves every CTA at least one k-tile; 1 otherwise.
int clusterk_slices(long long tiles, int KT, int sms) {
    int S = 8;
    while (S > 1 && (tiles * S > sms || S > KT)) S /= 2;
    return S;
}

namespace {

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
    {"ck_tma_128x256_k64_s2", 128, 256, 2, 4, 2, kLoaderTma, kScheduleClusterK},
    {"ck_tma_256x128_k64_s2", 256, 128, 4, 2, 2, kLoaderTma, kScheduleClusterK},
    {"packed_ck_tma_128x256_k64_s2", 128, 256, 2, 4, 2, kLoaderTma, kScheduleClusterK},
    {"ck_tma_128x256_s4", 128, 256, 2, 4, 4, kLoaderTma, kScheduleClusterK},
    {"ck_tma_256x128_s4", 256, 128, 4, 2, 4, kLoaderTma, kScheduleClusterK},
};
constexpr int kNumConfigs = sizeof(kConfigs) / sizeof(kConfigs[0]);

bool packable(const SimtProblem &p);
cudaError_t launch_small_splitk(const SimtProblem &p, cudaStream_t stream, const char **detail);
cudaError_t launch_packed(int inner, const SimtProblem &p, cudaStream_t stream,
                          const char **detail);
bool stage_c(int id, const SimtProblem &p);
cudaError_t launch_staged_c(int id, const SimtProblem &p, cudaStream_t stream,
                            const char **detail);
cudaError_t launch_config(int id, const SimtProblem &p, cudaStream_t stream,
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
    if (id == 14 || id == 15 || id == 18 || id == 22) return packable(p);
    if (kConfigs[id].loader == kLoaderTma) return tma_ok(p);
    return true;
}

cudaError_t simt_launch(int id, const SimtProblem &p, cudaStream_t stream, const char **detail) {
    if (id < 0 || id >= kNumConfigs) {
        *detail = "unknown SIMT configuration";
        return cudaErrorInvalidValue;
    }
    return stage_c(id, p) ? launch_staged_c(id, p, stream, detail)
                          : launch_config(id, p, stream, detail);
}

namespace {

cudaError_t launch_config(int id, const SimtProblem &p, cudaStream_t stream,
                          const char **detail) {
    switch (id) {
        case 0: case 1: case 2: return simt_launch_dp(id, p, stream, detail);
        case 3: case 4: return simt_launch_dpcp(id, p, stream, detail);
        case 5: case 6: case 7: return simt_launch_sk(id, p, stream, detail);
        case 8: case 9: return simt_launch_sk128(id, p, stream, detail);
        case 10: return skinny_launch(kSkinnyTall, p, stream, detail);
        case 11: return skinny_launch(kSkinnyWide, p, stream, detail);
        case 12: case 13: return simt_launch_skcp(id, p, stream, detail);
        case 14: return launch_packed(5, p, stream, detail);
        case 15: return launch_packed(2, p, stream, detail);
        case 16: case 17: return simt_launch_sk64(id, p, stream, detail);
        case 18: return launch_packed(17, p, stream, detail);
        case 19: return launch_small_splitk(p, stream, detail);
        case 20: case 21: case 23: case 24: return simt_launch_ck(id, p, stream, detail);
        case 22: return launch_packed(20, p, stream, detail);
        default: *detail = "unknown SIMT configuration"; return cudaErrorInvalidValue;
    }
}

}  // namespace

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

// One operand to copy: rows x cols values (leading dimension lds, batch stride ss) into dst
// (leading dimension ldd, a multiple of 4, 16-byte aligned base; batch stride sd), by a grid of
// gx x gy CTAs (gx across a row, gy down the rows of every batch entry).
struct PackJob {
    const float *src;
    long long lds, ss;
    float *dst;
    long long ldd, sd;
    int rows, cols;
    int gx, gy;
};

PackJob pack_job(const float *src, long long lds, long long ss, float *dst, long long ldd,
                 long long sd, int rows, int cols, int batch) {
    const long long nrows = static_cast<long long>(rows) * batch;
    const int gx = static_cast<int>(std::max<long long>(1, std::min<long long>((cols + 1023) / 1024, 8)));
    // About 2,048 CTAs per operand, each looping over several rows: with one CTA per row the
    // CTAs spent most of their time being scheduled (4095 x 3001 x 1537, both copies: 19.3 us
    // with a CTA per row, 15.4 us so).
    const int gy = static_cast<int>(std::max<long long>(1, std::min<long long>(nrows, 2048 / gx)));
    return {src, lds, ss, dst, ldd, sd, rows, cols, gx, gy};
}

// Both operands in one launch, so that the two copies stream at once: CTAs [0, gx0 * gy0) copy
// the first job, the rest the second. Rows run down the job's gy (batch entries stacked),
// columns across its gx, four consecutive columns per thread: four scalar loads from the
// unaligned source row (a warp's loads still cover 512 contiguous bytes) and one 16-byte store
// into the aligned copy.
__global__ void pack_rows_kernel(const PackJob j0, const PackJob j1, int batch) {
    // the GEMM that reads the copies may start its prologue now (it waits for this grid)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    long long bid = blockIdx.x;
    const long long blocks0 = static_cast<long long>(j0.gx) * j0.gy;
    const bool first = bid < blocks0;
    const PackJob &j = first ? j0 : j1;
    if (!first) bid -= blocks0;
    const int bx = static_cast<int>(bid % j.gx);
    const long long by = bid / j.gx;
    const long long nrows = static_cast<long long>(j.rows) * batch;
    const int c4 = j.cols & ~3;
    for (long long gr = by; gr < nrows; gr += j.gy) {
        const long long b = gr / j.rows, r = gr - b * j.rows;
        const float *s = j.src + b * j.ss + r * j.lds;
        float *d = j.dst + b * j.sd + r * j.ldd;
        for (int c = 4 * (bx * blockDim.x + threadIdx.x); c < c4; c += 4 * j.gx * blockDim.x) {
            const float4 v = make_float4(__ldcs(s + c), __ldcs(s + c + 1), __ldcs(s + c + 2),
                                         __ldcs(s + c + 3));
            *reinterpret_cast<float4 *>(d + c) = v;
        }
        for (int c = c4 + bx * blockDim.x + threadIdx.x; c < j.cols; c += j.gx * blockDim.x)
            d[c] = s[c];
    }
}

// Grid of the staged-C pass: up to 8 CTAs of 1,024 columns across a row, a CTA per row (more
// CTAs in flight keep this bandwidth-bound pass at the copy rate; capping the grid at 2,048
// CTAs made it 6% slower).
dim3 rows_grid(long long rows, int cols) {
    const unsigned x = static_cast<unsigned>(std::min<long long>((cols + 1023) / 1024, 8));
    const unsigned y = static_cast<unsigned>(std::min<long long>(rows, 65535));
    return dim3(x > 0 ? x : 1, y);
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
constexpr int kSlotStagedC = 4;       // the product of a staged-C call (stage_c)

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

// ---- small problems: 64 x 64 tiles, K split over the warps of a CTA and over CTAs ------------
//
// For problems of a few tiles the large kernels leave most SMs idle and spend their time on
// cold instruction fetch of a fully unrolled loop. Here a CTA of kSmallWarps warps computes one
// 64 x 64 tile: each warp takes its own slice of K through its own two-stage cp.async ring (any
// alignment), with the same 8 x 16 thread tile and fragment layout and a rolled k loop; the
// warps then add their partial tiles through shared memory, warp w the rows [8w/W, 8(w+1)/W)
// of every thread tile, in warp order. With more than one CTA per tile (the grid's y), each CTA
// stores its sum, and the CTA that finishes a tile last (an atomic count per tile; nothing
// waits) adds the CTAs' sums in CTA order and applies the epilogue, then resets the count for
// the next call. Results do not depend on which CTA finishes when. The kernel is compiled per
// loader form (16- or 4-byte copies of A and of B) and per epilogue form (plain or fused), so
// each instance carries only the code it runs: at this size a cold instruction cache is a large
// share of the time.

constexpr int kSmallWarps = 4;
constexpr int kSmallStageFloats = 64 * BK + BK * 64;  // one stage: 16 KiB
constexpr size_t kSmallSmem = static_cast<size_t>(kSmallWarps) * 2 * kSmallStageFloats * 4;

struct SmallParams {
    KParams k;
    int ctas;                // CTAs per tile (grid y)
    int kt_per_slice;        // 32-wide k-tiles per warp
    float4 *partials;        // [tile][cta][32 x 32 float4]
    unsigned int *counters;  // [tile]: CTAs finished
};

template <int AV, int BV, int FUSED>
__global__ void __launch_bounds__(kSmallWarps * 32) small_splitk_kernel(const SmallParams sp) {
    const KParams &p = sp.k;
    extern __shared__ __align__(16) float small_smem[];  // [warp][2 stages][kSmallStageFloats]
    __shared__ unsigned int s_last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tile = blockIdx.x, cta = blockIdx.y;
    const int tiles_per_batch = p.tiles_m * p.tiles_n;
    const int b = tile / tiles_per_batch;
    int tm, tn;
    tile_coords(tile - b * tiles_per_batch, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    const int m0 = tm * 64, n0 = tn * 64;
    const int KT = (p.K + BK - 1) / BK;
    const int slice = cta * kSmallWarps + warp;
    const int kt0 = min(KT, slice * sp.kt_per_slice);
    const int kt1 = min(KT, kt0 + sp.kt_per_slice);
    const float *Ab = p.A + static_cast<long long>(b) * p.sA;
    const float *Bb = p.B + static_cast<long long>(b) * p.sB;
    const int tr = lane >> 2, tc = lane & 3;
    float *ring = small_smem + warp * 2 * kSmallStageFloats;

    float2 acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[r][j] = make_float2(0.0f, 0.0f);

    if (kt0 < kt1)
        cp_async_stage<64, 64, 32, AV, BV>(ring, ring + 64 * BK, p, Ab, Bb, m0, n0, kt0 * BK, lane);
    cp_async_commit();
#pragma unroll 1
    for (int kt = kt0; kt < kt1; ++kt) {
        float *st = ring + ((kt - kt0) & 1) * kSmallStageFloats;
        float *nx = ring + (((kt - kt0) & 1) ^ 1) * kSmallStageFloats;
        if (kt + 1 < kt1)
            cp_async_stage<64, 64, 32, AV, BV>(nx, nx + 64 * BK, p, Ab, Bb, m0, n0, (kt + 1) * BK,
                                               lane);
        cp_async_commit();
        cp_async_wait<1>();
        __syncwarp();  // k-tile kt landed for the whole warp
        compute_ktile<64, kOrderHalfSnake, 1>(st + tr * BK, tr, st + 64 * BK + 4 * tc, acc);
        __syncwarp();  // the stage is free for the load two k-tiles ahead
    }
    cp_async_wait<0>();
    __syncwarp();

    // This warp's partial tile into its own ring (16 KiB: one float4 per (j, lane)).
    float4 *part = reinterpret_cast<float4 *>(ring);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int r = j >> 2, q = j & 3;
        part[j * 32 + lane] = make_float4(acc[r][2 * q].x, acc[r][2 * q].y, acc[r][2 * q + 1].x,
                                          acc[r][2 * q + 1].y);
    }
    __syncthreads();  // every warp's partial tile is in shared memory

    // Warp w adds rows [r0, r1) of the thread tiles over the warps, in warp order.
    const int r0 = warp * 8 / kSmallWarps, r1 = (warp + 1) * 8 / kSmallWarps;
    const float4 *parts = reinterpret_cast<const float4 *>(small_smem);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        if (r < r0 || r >= r1) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = r * 4 + q;
            float4 sum = parts[j * 32 + lane];
#pragma unroll
            for (int w = 1; w < kSmallWarps; ++w) {
                const float4 v = parts[static_cast<size_t>(w) * 2 * kSmallStageFloats / 4 + j * 32 + lane];
                sum.x += v.x;
                sum.y += v.y;
                sum.z += v.z;
                sum.w += v.w;
            }
            acc[r][2 * q] = make_float2(sum.x, sum.y);
            acc[r][2 * q + 1] = make_float2(sum.z, sum.w);
        }
    }

    float *Cb = p.C + static_cast<long long>(b) * p.sC;
    if (sp.ctas == 1) {
        epilogue<1, FUSED>(p, Cb, m0 + tr, n0 + 4 * tc, acc, r0, r1);
        return;
    }
    // Several CTAs per tile: store this CTA's sums; the last CTA to finish adds them all.
    float4 *mine = sp.partials + (static_cast<size_t>(tile) * sp.ctas + cta) * 1024;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        if (r < r0 || r >= r1) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            mine[(r * 4 + q) * 32 + lane] = make_float4(acc[r][2 * q].x, acc[r][2 * q].y,
                                                        acc[r][2 * q + 1].x, acc[r][2 * q + 1].y);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = atomicAdd(&sp.counters[tile], 1u) == static_cast<unsigned int>(sp.ctas - 1);
    __syncthreads();
    if (!s_last) return;  // not the last CTA of this tile to finish
    __threadfence();
    const float4 *base = sp.partials + static_cast<size_t>(tile) * sp.ctas * 1024;
#pragma unroll 1
    for (int c = 0; c < sp.ctas; ++c) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            if (r < r0 || r >= r1) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 v = __ldcg(base + static_cast<size_t>(c) * 1024 + (r * 4 + q) * 32 + lane);
                if (c == 0) {
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
    }
    if (threadIdx.x == 0) sp.counters[tile] = 0u;  // ready for the next launch on this stream
    epilogue<1, FUSED>(p, Cb, m0 + tr, n0 + 4 * tc, acc, r0, r1);
}

// The instance for the problem's loader and epilogue forms, with its shared-memory limit set
// once per device.
template <int AV, int BV, int FUSED>
cudaError_t launch_small_instance(int dev, const SmallParams &sp, dim3 grid, cudaStream_t stream) {
    auto kernel = small_splitk_kernel<AV, BV, FUSED>;
    static std::once_flag once[kMaxDevices];
    static cudaError_t attr_err[kMaxDevices];
    std::call_once(once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmallSmem));
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];
    kernel<<<grid, kSmallWarps * 32, kSmallSmem, stream>>>(sp);
    return cudaGetLastError();
}

cudaError_t launch_small_splitk(const SimtProblem &p, cudaStream_t stream, const char **detail) {
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
    // Warp slices of K: a CTA's warps share a tile's k-tiles; more CTAs per tile (one CTA per
    // SM, its shared memory is 128 KiB) only once a warp would run more than kSmallKtPerWarp
    // k-tiles, as many as the SMs hold next to the other tiles, at most 16. A second CTA costs a
    // pass of partial sums through global memory, measured between one and two k-tiles of a
    // warp (256^3: one CTA per tile 15.9 us against two 17.2 us; 512^3: two CTAs 20.8 us
    // against one 22.8 us).
    constexpr long long kSmallKtPerWarp = 2;
    const long long KT = std::max<long long>(1, (p.K + BK - 1) / BK);
    const int sms = std::max(1, device_sms(dev));
    long long ctas = std::max<long long>(1, std::min<long long>(sms / tiles, 16));
    ctas = std::min<long long>(ctas, (KT + kSmallWarps * kSmallKtPerWarp - 1) /
                                         (kSmallWarps * kSmallKtPerWarp));
    const long long per = (KT + ctas * kSmallWarps - 1) / (ctas * kSmallWarps);
    ctas = (KT + per * kSmallWarps - 1) / (per * kSmallWarps);  // no CTA without k-tiles
    if (ctas < 1) ctas = 1;
    sp.ctas = static_cast<int>(ctas);
    sp.kt_per_slice = static_cast<int>(per);
    sp.partials = nullptr;
    sp.counters = nullptr;
    if (ctas > 1) {
        // The counts live in their own allocation: zeroed whenever it is (re)allocated, and
        // left at zero by every launch (the last CTA of each tile resets its count), so any
        // later launch on this stream, of any tile count that fits, starts from zeros.
        float *cnt = nullptr, *ws = nullptr;
        bool fresh = false;
        const size_t count_bytes = static_cast<size_t>(tiles) * sizeof(unsigned int);
        err = pack_workspace(dev, stream, kSlotSplitKCount, count_bytes, &cnt, &fresh);
        if (err == cudaSuccess && fresh) err = cudaMemsetAsync(cnt, 0, count_bytes, stream);
        if (err == cudaSuccess)
            err = pack_workspace(dev, stream, kSlotSplitK,
                                 static_cast<size_t>(tiles) * ctas * 1024 * sizeof(float4), &ws);
        if (err != cudaSuccess) {
            *detail = "split-K workspace allocation failed";
            return err;
        }
        sp.counters = reinterpret_cast<unsigned int *>(cnt);
        sp.partials = reinterpret_cast<float4 *>(ws);
    }
    const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(ctas));
    const bool fused = p.bias != nullptr || p.act != kActNone;
    const int form = (kp.a_vec4 ? 4 : 0) + (kp.b_vec4 ? 2 : 0) + (fused ? 1 : 0);
    switch (form) {
        case 0: err = launch_small_instance<0, 0, 0>(dev, sp, grid, stream); break;
        case 1: err = launch_small_instance<0, 0, 1>(dev, sp, grid, stream); break;
        case 2: err = launch_small_instance<0, 1, 0>(dev, sp, grid, stream); break;
        case 3: err = launch_small_instance<0, 1, 1>(dev, sp, grid, stream); break;
        case 4: err = launch_small_instance<1, 0, 0>(dev, sp, grid, stream); break;
        case 5: err = launch_small_instance<1, 0, 1>(dev, sp, grid, stream); break;
        case 6: err = launch_small_instance<1, 1, 0>(dev, sp, grid, stream); break;
        default: err = launch_small_instance<1, 1, 1>(dev, sp, grid, stream); break;
    }
    if (err != cudaSuccess) *detail = "small split-K kernel launch failed";
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
        PackJob jobs[2];
        int njobs = 0;
        if (packA) {
            jobs[njobs++] = pack_job(p.A, p.lda, p.strideA, ws, ldA, elemsA, p.M, p.K, p.batch);
            q.A = ws;
            q.lda = ldA;
            q.strideA = p.batch > 1 ? elemsA : 0;
        }
        if (packB) {
            float *wb = ws + elemsA * p.batch;
            jobs[njobs++] = pack_job(p.B, p.ldb, p.strideB, wb, ldB, elemsB, p.K, p.N, p.batch);
            q.B = wb;
            q.ldb = ldB;
            q.strideB = p.batch > 1 ? elemsB : 0;
        }
        long long blocks = 0;
        for (int i = 0; i < njobs; ++i) blocks += static_cast<long long>(jobs[i].gx) * jobs[i].gy;
        pack_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(jobs[0], jobs[njobs - 1],
                                                                           p.batch);
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
    q.pdl = packA || packB;  // the persistent kernels overlap their prologue with the copy
    return launch_config(inner, q, stream, detail);
}

// ---- C that the epilogue cannot read with 16-byte loads, beta != 0 ------------------------------
//
// With an unaligned C (odd ldc, say) the tile epilogue reads C with 4-byte loads, one memory
// round trip per few values, while its warps wait (4095 x 3001 x 1537: 61 us of 742). For
// large problems the product is computed instead into an aligned scratch D with the beta = 0
// epilogue (alpha = 1, no bias or activation: D holds the fp32 accumulators as they are), and a
// streaming pass applies the caller's epilogue to C: the same expression on the same fp32
// values, so the result is bit-identical to the in-kernel epilogue.
constexpr long long kStageCMinElems = 1LL << 22;

// Rows over the grid's y dimension (batch entries stacked), four consecutive columns per
// thread: one 16-byte load of D (its leading dimension is a multiple of 4; a row's last,
// partial group is read value by value, so the scratch's unwritten padding is never read),
// the C values loaded before any store.
__global__ void apply_staged_c_kernel(const float *__restrict__ D, long long ldd, long long sd,
                                      float *__restrict__ C, long long ldc, long long sc,
                                      int rows, int cols, int batch, float alpha, float beta,
                                      const float *__restrict__ bias, int act) {
    // launched as a programmatic dependent of the GEMM: D is read only once that grid is done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long nrows = static_cast<long long>(rows) * batch;
    const bool fused = bias != nullptr || act != kActNone;
    for (long long gr = blockIdx.y; gr < nrows; gr += gridDim.y) {
        const long long b = gr / rows, r = gr - b * rows;
        const float *d = D + b * sd + r * ldd;
        float *c = C + b * sc + r * ldc;
        for (int j = 4 * (blockIdx.x * blockDim.x + threadIdx.x); j < cols;
             j += 4 * gridDim.x * blockDim.x) {
            const int n = cols - j < 4 ? cols - j : 4;
            float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (n == 4) {
                const float4 v4 = __ldcs(reinterpret_cast<const float4 *>(d + j));
                v[0] = v4.x;
                v[1] = v4.y;
                v[2] = v4.z;
                v[3] = v4.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (e < n) v[e] = d[j + e];
            }
            float cv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < n) cv[e] = c[j + e];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < n)
                    c[j + e] = fused ? epilogue_apply(v[e], alpha, beta, bias, j + e, act, cv[e])
                                     : fmaf(alpha, v[e], beta * cv[e]);
        }
    }
}

bool stage_c(int id, const SimtProblem &p) {
    if (p.beta == 0.0f || operand_vec4(p.C, p.ldc, p.strideC, p.batch)) return false;
    if (id == 10 || id == 11 || id == 19) return false;  // skinny and small-problem kernels
    return static_cast<long long>(p.M) * p.N * p.batch >= kStageCMinElems;
}

cudaError_t launch_staged_c(int id, const SimtProblem &p, cudaStream_t stream,
                            const char **detail) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) {
        *detail = "cudaGetDevice failed";
        return err;
    }
    const long long ldd = (static_cast<long long>(p.N) + 3) / 4 * 4;
    const long long elems = static_cast<long long>(p.M) * ldd;
    float *D = nullptr;
    err = pack_workspace(dev, stream, kSlotStagedC, static_cast<size_t>(elems) * p.batch * 4, &D);
    if (err != cudaSuccess) {
        *detail = "staged-C workspace allocation failed";
        return err;
    }
    SimtProblem q = p;
    q.C = D;
    q.ldc = ldd;
    q.strideC = p.batch > 1 ? elems : 0;
    q.alpha = 1.0f;
    q.beta = 0.0f;
    q.bias = nullptr;
    q.act = kActNone;
    q.pdl_next = true;  // the pass below may begin its launch while the GEMM runs
    err = launch_config(id, q, stream, detail);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = rows_grid(static_cast<long long>(p.M) * p.batch, p.N);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, apply_staged_c_kernel, static_cast<const float *>(D), ldd,
                             elems, p.C, p.ldc, p.strideC, p.M, p.N, p.batch, p.alpha, p.beta,
                             p.bias, p.act);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) *detail = "staged-C epilogue launch failed";
    return err;
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
