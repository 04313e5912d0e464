// tf32x3_gemm.cu: tcgen05 3xTF32 path (kernel not built yet: reports unsupported).
#include "ptx.cuh"
#include "tf32x3_gemm.cuh"

namespace sg {

bool tf32x3_supports(const SimtProblem &) { return false; }

cudaError_t tf32x3_launch(const SimtProblem &, cudaStream_t, const char **detail) {
    *detail = "3xTF32 kernel not available";
    return cudaErrorNotSupported;
}

unsigned int tf32x3_take_fault_word(cudaStream_t) { return 0; }

}  // namespace sg
