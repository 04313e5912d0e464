// host_gemm.cuh: the product with host-memory operands (chunked, copies overlapping compute).
#pragma once

#include <cuda_runtime.h>

namespace sg {

struct HostProblem {
    long long M, N, K;
    float alpha, beta;
    const float *A;
    long long lda;
    const float *B;
    long long ldb;
    float *C;
    long long ldc;
};

// A device product on `stream` (device pointers); returns cudaSuccess or an error with
// `detail` set.
using DeviceGemmFn = cudaError_t (*)(long long M, long long N, long long K, float alpha,
                                     const float *A, long long lda, const float *B,
                                     long long ldb, float beta, float *C, long long ldc,
                                     cudaStream_t stream, const char **detail);

// Runs the host-memory product through device buffers; returns when C is back in host memory.
cudaError_t host_gemm(const HostProblem &p, cudaStream_t stream, DeviceGemmFn gemm,
                      const char **detail);

// Frees the per-device buffers of the host-memory path.
cudaError_t release_host_buffers();

}  // namespace sg
