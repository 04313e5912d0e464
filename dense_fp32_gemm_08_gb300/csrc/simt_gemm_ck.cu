// simt_gemm_ck.cu: the cluster split-K SIMT configurations for grids of under one wave (each
// output tile split along K over a thread-block cluster, reduced through distributed shared
// memory).
#include "simt_kernels.cuh"

namespace sg {

cudaError_t simt_launch_ck(int id, const SimtProblem &p, cudaStream_t stream, const char **detail) {
    switch (id) {
        case 20: return launch_clusterk<128, 256, 2, 4, 2, 2>(p, stream, detail);
        case 21: return launch_clusterk<256, 128, 4, 2, 2, 2>(p, stream, detail);
        case 23: return launch_clusterk<128, 256, 2, 4, 4, 1>(p, stream, detail);
        case 24: return launch_clusterk<256, 128, 4, 2, 4, 1>(p, stream, detail);
        default: *detail = "configuration not in this kernel unit"; return cudaErrorInvalidValue;
    }
}

}  // namespace sg
