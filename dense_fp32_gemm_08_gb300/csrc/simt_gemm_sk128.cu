// simt_gemm_sk128.cu: the persistent stream-K SIMT configurations with 128 x 128 tiles (two
// four-warp CTAs per SM).
#include "simt_kernels.cuh"

namespace sg {

cudaError_t simt_launch_sk128(int id, const SimtProblem &p, cudaStream_t stream, const char **detail) {
    switch (id) {
        case 8: return launch_persistent<128, 128, 2, 2, 3, 255>(kScheduleStreamK, p, stream, detail);
        case 9: return launch_persistent<128, 128, 2, 2, 4, 248>(kScheduleStreamK, p, stream, detail);
        default: *detail = "configuration not in this kernel unit"; return cudaErrorInvalidValue;
    }
}

}  // namespace sg
