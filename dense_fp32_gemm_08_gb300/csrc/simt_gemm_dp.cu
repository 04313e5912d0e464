// simt_gemm_dp.cu: the data-parallel SIMT configurations with the TMA loader (one CTA per
// output tile).
#include "simt_kernels.cuh"

namespace sg {

cudaError_t simt_launch_dp(int id, const SimtProblem &p, cudaStream_t stream, const char **detail) {
    switch (id) {
        case 0: return launch_impl<128, 256, 2, 4, 4, kLoaderTma>(id, p, stream, detail);
        case 1: return launch_impl<256, 128, 4, 2, 4, kLoaderTma>(id, p, stream, detail);
        case 2: return launch_impl<128, 128, 2, 2, 3, kLoaderTma>(id, p, stream, detail);
        default: *detail = "configuration not in this kernel unit"; return cudaErrorInvalidValue;
    }
}

}  // namespace sg
