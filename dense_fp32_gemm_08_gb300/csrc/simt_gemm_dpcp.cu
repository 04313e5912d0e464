// simt_gemm_dpcp.cu: the data-parallel SIMT configurations with the cp.async loader (any
// alignment).
#include "simt_kernels.cuh"

namespace sg {

cudaError_t simt_launch_dpcp(int id, const SimtProblem &p, cudaStream_t stream, const char **detail) {
    switch (id) {
        case 3: return launch_impl<128, 256, 2, 4, 4, kLoaderCpAsync>(id, p, stream, detail);
        case 4: return launch_impl<128, 128, 2, 2, 3, kLoaderCpAsync>(id, p, stream, detail);
        default: *detail = "configuration not in this kernel unit"; return cudaErrorInvalidValue;
    }
}

}  // namespace sg
