// simt_gemm_sk.cu: the persistent stream-K SIMT configurations with 32-wide TMA stages and 8
// warps per CTA, and sgemm_noalloc, which runs the 128 x 256 one with its partial sums in a
// static device array.
#include "simt_kernels.cuh"

namespace sg {

cudaError_t simt_launch_sk(int id, const SimtProblem &p, cudaStream_t stream, const char **detail) {
    switch (id) {
        case 5: return launch_persistent<128, 256, 2, 4, 4>(kScheduleStreamK, p, stream, detail);
        case 6: return launch_persistent<128, 256, 2, 4, 4>(kSchedulePersistentDP, p, stream, detail);
        case 7: return launch_persistent<256, 128, 4, 2, 4>(kScheduleStreamK, p, stream, detail);
        default: *detail = "configuration not in this kernel unit"; return cudaErrorInvalidValue;
    }
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
    pp.chain = 0;
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

}  // namespace sg
