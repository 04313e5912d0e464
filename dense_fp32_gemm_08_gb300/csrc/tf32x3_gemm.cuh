// tf32x3_gemm.cuh: the tcgen05 tensor-core path that emulates fp32 with three TF32 products.
#pragma once

#include <cuda_runtime.h>

#include "simt_gemm.cuh"

namespace sg {

// True when the 3xTF32 kernel can run this problem (any alignment: the split pre-pass reads
// A and B with plain loads; at most 65535 batch entries).
bool tf32x3_supports(const SimtProblem &p);

cudaError_t tf32x3_launch(const SimtProblem &p, cudaStream_t stream, const char **detail);

// One TF32 product per multiply-add (operands rounded to TF32): the fast, lower-accuracy mode.
cudaError_t tf32_launch(const SimtProblem &p, cudaStream_t stream, const char **detail);


// Frees the per-(device, stream) workspaces holding the split operands.
cudaError_t tf32x3_release_workspaces();

}  // namespace sg
