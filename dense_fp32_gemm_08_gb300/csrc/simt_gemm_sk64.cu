// simt_gemm_sk64.cu: the persistent stream-K SIMT configurations whose pipeline stages hold two
// 32-wide k sub-tiles (one CTA barrier and one TMA refill per 64 values of k).
#include "simt_kernels.cuh"

namespace sg {

cudaError_t simt_launch_sk64(int id, const SimtProblem &p, cudaStream_t stream, const char **detail) {
    // K mod 64 in [1, 32]: the last stage's second sub-tile is all padding (the KTAIL instance)
    const bool tail = p.K % 64 != 0 && p.K % 64 <= 32;
    switch (id) {
        case 16:
            return tail ? launch_persistent<128, 256, 2, 4, 2, 255, kLoaderTma, 2, 1>(kScheduleStreamK, p, stream, detail)
                        : launch_persistent<128, 256, 2, 4, 2, 255, kLoaderTma, 2, 0>(kScheduleStreamK, p, stream, detail);
        case 17:
            return tail ? launch_persistent<256, 128, 4, 2, 2, 255, kLoaderTma, 2, 1>(kScheduleStreamK, p, stream, detail)
                        : launch_persistent<256, 128, 4, 2, 2, 255, kLoaderTma, 2, 0>(kScheduleStreamK, p, stream, detail);
        default: *detail = "configuration not in this kernel unit"; return cudaErrorInvalidValue;
    }
}

}  // namespace sg
