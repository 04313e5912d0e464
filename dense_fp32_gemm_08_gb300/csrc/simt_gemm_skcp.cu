// simt_gemm_skcp.cu: the persistent stream-K SIMT configurations with the cp.async loader (any
// alignment).
#include "simt_kernels.cuh"

namespace sg {

cudaError_t simt_launch_skcp(int id, const SimtProblem &p, cudaStream_t stream, const char **detail) {
    switch (id) {
        case 12: return launch_persistent<128, 256, 2, 4, 4, 255, kLoaderCpAsync>(kScheduleStreamK, p, stream, detail);
        case 13: return launch_persistent<256, 128, 4, 2, 4, 255, kLoaderCpAsync>(kScheduleStreamK, p, stream, detail);
        default: *detail = "configuration not in this kernel unit"; return cudaErrorInvalidValue;
    }
}

}  // namespace sg
