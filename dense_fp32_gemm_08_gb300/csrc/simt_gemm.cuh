// simt_gemm.cuh: host-visible description of the FP32 SIMT kernels (tile configurations and
// the launch entry used by the dispatcher in sgemm_api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sg {

// How A and B tiles travel from global to shared memory.
enum LoaderKind : int {
    kLoaderTma = 0,      // cp.async.bulk.tensor (TMA), 16-byte aligned operands only
    kLoaderCpAsync = 1,  // cp.async, 16-byte chunks where an operand allows, else 4-byte
};

// Order in which tiles are assigned to CTAs.
enum ScheduleKind : int {
    kScheduleSkinny = -1,       // not a tiled kernel: a bandwidth kernel (skinny_gemm.cu)
    kScheduleDataParallel = 0,  // one CTA per output tile (grouped raster order)
    kScheduleStreamK = 1,       // persistent CTAs, the last one-to-two waves split along K
    kSchedulePersistentDP = 2,  // persistent CTAs, whole tiles round-robin
    kScheduleClusterK = 3,      // each tile split along K over a thread-block cluster
};

struct SimtConfig {
    const char *name;
    int bm, bn;      // CTA tile
    int warps_m, warps_n;
    int stages;      // depth of the shared-memory ring
    int loader;      // LoaderKind
    int schedule;    // ScheduleKind
};

// One problem (or one batch of equally shaped problems) as the kernels see it.
struct SimtProblem {
    int M, N, K;
    float alpha, beta;
    const float *A;
    const float *B;
    float *C;
    long long lda, ldb, ldc;
    long long strideA, strideB, strideC;  // element strides between batch entries
    int batch;
    bool transA = false;  // A stored K x M (op(A) = A^T); the tile kernels take false only
    bool transB = false;  // B stored N x K (op(B) = B^T); the tile kernels take false only
    const float *bias = nullptr;  // fused epilogue: per-column bias (N values), or none
    int act = 0;                  // fused epilogue: Activation (epilogue.cuh)
    // The library's own chaining of kernels on one stream (programmatic dependent launch);
    // callers leave both false. pdl: the launch follows a library kernel that lets it start
    // early, and the persistent kernels wait for that kernel's completion before they read
    // memory. pdl_next: a library kernel launched after this one may start early (it waits
    // for this one's completion in the same way).
    bool pdl = false;
    bool pdl_next = false;
};

int simt_num_configs();

// Multiprocessors of the calling thread's current device (queried once per device), or 0 when
// there is no device to query.
int simt_device_sms();
const SimtConfig &simt_config(int id);

// True when config `id` can run this problem (alignment needs of its loader).
bool simt_config_supports(int id, const SimtProblem &p);

// Launches config `id` on `stream`. Returns cudaSuccess or the launch / setup error;
// `detail` receives a static description of a failing step.
cudaError_t simt_launch(int id, const SimtProblem &p, cudaStream_t stream, const char **detail);


// Frees every per-device workspace the SIMT kernels allocated (stream-K partial tiles).
cudaError_t release_workspaces();

// Frees the per-(device, stream) copies of operands repacked for TMA.
cudaError_t release_pack_workspaces();

// Turns a problem with transposed operands into the same product with row-major,
// non-transposed, 16-byte aligned copies of those operands (written on `stream` into a
// per-(device, stream) workspace). `q` receives the rewritten problem.
cudaError_t simt_untranspose(const SimtProblem &p, cudaStream_t stream, SimtProblem *q,
                             const char **detail);

// Launches a one-thread kernel whose bounded wait can never be satisfied (which = 0: an
// mbarrier, 1: a flag word), to exercise the timeout path.
cudaError_t simt_selftest_wait(int which, cudaStream_t stream);

// The stream-K 128 x 256 kernel with its partial sums in a static device array: allocates
// nothing. Returns cudaErrorNotSupported (with `detail`) when the operands are not TMA-aligned
// or the call needs more partial-sum slots than the array holds.
cudaError_t simt_launch_noalloc(const SimtProblem &p, cudaStream_t stream, const char **detail);

}  // namespace sg
