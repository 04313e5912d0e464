// skinny_gemm.cuh: bandwidth kernels for products with one output dimension of at most 8.
#pragma once

#include <cuda_runtime.h>

#include "simt_gemm.cuh"

namespace sg {

using SkinnyProblem = SimtProblem;

enum SkinnyKind : int {
    kSkinnyTall = 0,  // N <= 8: stream A, one warp per row
    kSkinnyWide = 1,  // M <= 8: stream B, 128 columns per CTA, K split over an 8-CTA cluster
};

// True when kernel `kind` can run the problem.
bool skinny_supports(int kind, const SkinnyProblem &p);

cudaError_t skinny_launch(int kind, const SkinnyProblem &p, cudaStream_t stream,
                          const char **detail);

}  // namespace sg
