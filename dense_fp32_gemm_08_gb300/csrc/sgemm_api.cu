// sgemm_api.cu: the C ABI (include/sgemm.h): argument checks, fast exits, kernel choice and
// status reporting. Every compute step runs in the CUDA kernels of this library.
#include "sgemm.h"

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "config_table.h"
#include "epilogue.cuh"
#include "host_gemm.cuh"
#include "ptx.cuh"
#include "simt_gemm.cuh"
#include "tf32x3_gemm.cuh"

namespace sg {
namespace {
std::mutex &fault_reader_mutex() {
    static std::mutex m;
    return m;
}
std::vector<FaultWordReader> &fault_readers() {
    static std::vector<FaultWordReader> v;
    return v;
}
}  // namespace

void register_fault_word_reader(FaultWordReader reader) {
    std::lock_guard<std::mutex> lock(fault_reader_mutex());
    fault_readers().push_back(reader);
}

unsigned int take_fault_words(cudaStream_t stream) {
    std::vector<FaultWordReader> readers;
    {
        std::lock_guard<std::mutex> lock(fault_reader_mutex());
        readers = fault_readers();
    }
    unsigned int word = 0;
    for (FaultWordReader read : readers) word |= read(stream);
    return word;
}
}  // namespace sg

namespace {

thread_local char t_last_error[256] = "";

sgemm_status_t fail(sgemm_status_t st, const char *what) {
    std::snprintf(t_last_error, sizeof(t_last_error), "%s", what);
    return st;
}

sgemm_status_t fail_cuda(const char *what, cudaError_t err) {
    std::snprintf(t_last_error, sizeof(t_last_error), "%s: %s", what, cudaGetErrorString(err));
    return SGEMM_ERR_LAUNCH;
}

constexpr long long kMaxDim = 0x7fffffffLL;  // kernels index M, N, K with 32-bit ints

std::atomic<int> g_forced_config{-2};  // -2: environment not read yet, -1: automatic

int forced_config() {
    int v = g_forced_config.load(std::memory_order_relaxed);
    if (v == -2) {
        const char *env = std::getenv("SGEMM_FORCE_CONFIG");
        int want = -1;
        if (env && *env) {
            char *end = nullptr;
            long id = std::strtol(env, &end, 10);
            if (end && *end == '\0' && id >= 0 && id < sg::simt_num_configs()) want = (int)id;
        }
        int expected = -2;
        g_forced_config.compare_exchange_strong(expected, want);
        v = g_forced_config.load(std::memory_order_relaxed);
    }
    return v;
}

bool log_enabled() {
    static const bool on = [] {
        const char *env = std::getenv("SGEMM_LOG");
        return env && *env && std::strcmp(env, "0") != 0;
    }();
    return on;
}

// C = beta * C (zeros when beta == 0, C not read then), the whole product when alpha == 0 or
// K == 0; with a fused epilogue, C = act(bias) + beta * C. Rows over the grid's y dimension
// (batch entries stacked), columns over threads.
__global__ void scale_c_kernel(float *C, long long M, long long N, long long ldc,
                               long long strideC, long long batch, float beta,
                               const float *bias, int act) {
    const long long nrows = M * batch;
    const bool fused = bias != nullptr || act != sg::kActNone;
    for (long long gr = blockIdx.y; gr < nrows; gr += gridDim.y) {
        const long long b = gr / M, r = gr - b * M;
        float *row = C + b * strideC + r * ldc;
        for (long long c = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; c < N;
             c += static_cast<long long>(gridDim.x) * blockDim.x) {
            if (fused)
                row[c] = sg::epilogue_value(0.0f, 0.0f, beta, bias, static_cast<int>(c), act,
                                            row + c);
            else
                row[c] = beta == 0.0f ? 0.0f : beta * row[c];
        }
    }
}

struct Args {
    long long M, N, K;
    float alpha, beta;
    const float *A;
    long long lda, sA;
    const float *B;
    long long ldb, sB;
    float *C;
    long long ldc, sC;
    long long batch;
    bool ta = false, tb = false;  // A stored K x M, B stored N x K
    const float *bias = nullptr;  // fused epilogue
    int act = 0;
};

// Checks shared by every entry point. Returns SGEMM_OK when the arguments are valid.
sgemm_status_t validate(const Args &a) {
    if (a.M < 0 || a.N < 0 || a.K < 0) return fail(SGEMM_ERR_INVALID_VALUE, "M, N and K must be >= 0");
    if (a.batch < 0) return fail(SGEMM_ERR_INVALID_VALUE, "batch must be >= 0");
    const long long acols = a.ta ? a.M : a.K, bcols = a.tb ? a.K : a.N;
    if (a.lda < (acols > 1 ? acols : 1))
        return fail(SGEMM_ERR_INVALID_VALUE, a.ta ? "lda < max(1, M) (A transposed)" : "lda < max(1, K)");
    if (a.ldb < (bcols > 1 ? bcols : 1))
        return fail(SGEMM_ERR_INVALID_VALUE, a.tb ? "ldb < max(1, K) (B transposed)" : "ldb < max(1, N)");
    if (a.ldc < (a.N > 1 ? a.N : 1)) return fail(SGEMM_ERR_INVALID_VALUE, "ldc < max(1, N)");
    if (a.sA < 0 || a.sB < 0 || a.sC < 0)
        return fail(SGEMM_ERR_INVALID_VALUE, "batch strides must be >= 0");
    if (a.M == 0 || a.N == 0 || a.batch == 0) return SGEMM_OK;
    if (a.batch > 1 && a.sC < a.M * a.ldc)
        return fail(SGEMM_ERR_INVALID_VALUE, "strideC < M * ldc: batch outputs would overlap");
    if (!a.C) return fail(SGEMM_ERR_INVALID_VALUE, "C is NULL");
    const bool reads_ab = a.alpha != 0.0f && a.K > 0;
    if (reads_ab && (!a.A || !a.B)) return fail(SGEMM_ERR_INVALID_VALUE, "A or B is NULL");
    return SGEMM_OK;
}

bool is_noop(const Args &a) { return a.M == 0 || a.N == 0 || a.batch == 0; }

sgemm_status_t check_limits(const Args &a) {
    if (a.M > kMaxDim || a.N > kMaxDim || a.K > kMaxDim || a.batch > kMaxDim)
        return fail(SGEMM_ERR_UNSUPPORTED, "a dimension exceeds 2^31 - 1");
    return SGEMM_OK;
}

sgemm_status_t run_scale(const Args &a, cudaStream_t stream) {
    const long long nrows = a.M * a.batch;
    const dim3 grid(static_cast<unsigned>((a.N + 255) / 256 < 8 ? (a.N + 255) / 256 : 8),
                    static_cast<unsigned>(nrows < 65535 ? nrows : 65535));
    scale_c_kernel<<<grid, 256, 0, stream>>>(a.C, a.M, a.N, a.ldc, a.sC, a.batch, a.beta, a.bias,
                                             a.act);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return fail_cuda("scale kernel launch", err);
    return SGEMM_OK;
}

sg::SimtProblem to_problem(const Args &a) {
    sg::SimtProblem p;
    p.M = static_cast<int>(a.M);
    p.N = static_cast<int>(a.N);
    p.K = static_cast<int>(a.K);
    p.alpha = a.alpha;
    p.beta = a.beta;
    p.A = a.A;
    p.B = a.B;
    p.C = a.C;
    p.lda = a.lda;
    p.ldb = a.ldb;
    p.ldc = a.ldc;
    p.strideA = a.batch > 1 ? a.sA : 0;
    p.strideB = a.batch > 1 ? a.sB : 0;
    p.strideC = a.batch > 1 ? a.sC : 0;
    p.batch = static_cast<int>(a.batch);
    p.transA = a.ta;
    p.transB = a.tb;
    p.bias = a.bias;
    p.act = a.act;
    return p;
}

int choose_simt(const sg::SimtProblem &p) {
    const int forced = forced_config();
    if (forced >= 0 && sg::simt_config_supports(forced, p)) return forced;
    return sg::table_choose(p, sg::simt_device_sms());
}

sgemm_status_t run_simt(const Args &a, cudaStream_t stream) {
    sg::SimtProblem p = to_problem(a);
    if (p.transA || p.transB) {  // the tile kernels read op(A), op(B) row-major
        const char *detail = "";
        sg::SimtProblem q;
        cudaError_t err = sg::simt_untranspose(p, stream, &q, &detail);
        if (err != cudaSuccess) return fail_cuda(detail, err);
        p = q;
    }
    const int id = choose_simt(p);
    if (log_enabled())
        std::fprintf(stderr, "[sgemm] M=%lld N=%lld K=%lld batch=%lld -> %s\n", a.M, a.N, a.K,
                     a.batch, sg::simt_config(id).name);
    const char *detail = "";
    cudaError_t err = sg::simt_launch(id, p, stream, &detail);
    if (err != cudaSuccess) return fail_cuda(detail, err);
    return SGEMM_OK;
}

enum Path { kPathSimt, kPathTf32x3, kPathTf32 };

sgemm_status_t run_tensor(const Args &a, cudaStream_t stream, Path path) {
    const sg::SimtProblem p = to_problem(a);
    if (!sg::tf32x3_supports(p))
        return fail(SGEMM_ERR_UNSUPPORTED, "the TF32 paths take at most 65535 batch entries");
    const char *detail = "";
    cudaError_t err = path == kPathTf32 ? sg::tf32_launch(p, stream, &detail)
                                        : sg::tf32x3_launch(p, stream, &detail);
    if (err != cudaSuccess) return fail_cuda(detail, err);
    return SGEMM_OK;
}

bool have_device() {
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess;
}

sgemm_status_t dispatch(const Args &a, void *stream_ptr, Path path) {
    t_last_error[0] = '\0';
    sgemm_status_t st = validate(a);
    if (st != SGEMM_OK) return st;
    if (is_noop(a)) return SGEMM_OK;
    st = check_limits(a);
    if (st != SGEMM_OK) return st;
    if (!have_device()) return fail(SGEMM_ERR_UNSUPPORTED, "no CUDA device available");
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (a.alpha == 0.0f || a.K == 0) return run_scale(a, stream);
    return path == kPathSimt ? run_simt(a, stream) : run_tensor(a, stream, path);
}

// Device product used by each chunk of the host-memory path (the SIMT path).
cudaError_t chunk_gemm(long long M, long long N, long long K, float alpha, const float *A,
                       long long lda, const float *B, long long ldb, float beta, float *C,
                       long long ldc, cudaStream_t stream, const char **detail) {
    Args a{M, N, K, alpha, beta, A, lda, 0, B, ldb, 0, C, ldc, 0, 1};
    const sgemm_status_t st = (alpha == 0.0f || K == 0) ? run_scale(a, stream) : run_simt(a, stream);
    if (st != SGEMM_OK) {
        *detail = "a chunk's device product failed";
        return cudaErrorLaunchFailure;
    }
    return cudaSuccess;
}

}  // namespace

extern "C" {

sgemm_status_t sgemm(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                     const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                     void *stream) {
    Args a{M, N, K, alpha, beta, A, lda, 0, B, ldb, 0, C, ldc, 0, 1};
    return dispatch(a, stream, kPathSimt);
}

sgemm_status_t sgemm_strided_batched(int64_t M, int64_t N, int64_t K, float alpha,
                                     const float *A, int64_t lda, int64_t strideA,
                                     const float *B, int64_t ldb, int64_t strideB, float beta,
                                     float *C, int64_t ldc, int64_t strideC, int64_t batch,
                                     void *stream) {
    Args a{M, N, K, alpha, beta, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, batch};
    return dispatch(a, stream, kPathSimt);
}

sgemm_status_t sgemm_3xtf32(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                            int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                            int64_t ldc, void *stream) {
    Args a{M, N, K, alpha, beta, A, lda, 0, B, ldb, 0, C, ldc, 0, 1};
    return dispatch(a, stream, kPathTf32x3);
}

sgemm_status_t sgemm_3xtf32_strided_batched(int64_t M, int64_t N, int64_t K, float alpha,
                                            const float *A, int64_t lda, int64_t strideA,
                                            const float *B, int64_t ldb, int64_t strideB,
                                            float beta, float *C, int64_t ldc, int64_t strideC,
                                            int64_t batch, void *stream) {
    Args a{M, N, K, alpha, beta, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, batch};
    return dispatch(a, stream, kPathTf32x3);
}

sgemm_status_t sgemm_tf32(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                          int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                          int64_t ldc, void *stream) {
    Args a{M, N, K, alpha, beta, A, lda, 0, B, ldb, 0, C, ldc, 0, 1};
    return dispatch(a, stream, kPathTf32);
}

sgemm_status_t sgemm_tf32_strided_batched(int64_t M, int64_t N, int64_t K, float alpha,
                                          const float *A, int64_t lda, int64_t strideA,
                                          const float *B, int64_t ldb, int64_t strideB,
                                          float beta, float *C, int64_t ldc, int64_t strideC,
                                          int64_t batch, void *stream) {
    Args a{M, N, K, alpha, beta, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, batch};
    return dispatch(a, stream, kPathTf32);
}

sgemm_status_t sgemm_noalloc(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                             int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                             int64_t ldc, void *stream_ptr) {
    Args a{M, N, K, alpha, beta, A, lda, 0, B, ldb, 0, C, ldc, 0, 1};
    t_last_error[0] = '\0';
    sgemm_status_t st = validate(a);
    if (st != SGEMM_OK) return st;
    if (is_noop(a)) return SGEMM_OK;
    st = check_limits(a);
    if (st != SGEMM_OK) return st;
    if (!have_device()) return fail(SGEMM_ERR_UNSUPPORTED, "no CUDA device available");
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (a.alpha == 0.0f || a.K == 0) return run_scale(a, stream);  // allocates nothing either
    const char *detail = "";
    cudaError_t err = sg::simt_launch_noalloc(to_problem(a), stream, &detail);
    if (err == cudaErrorNotSupported) return fail(SGEMM_ERR_UNSUPPORTED, detail);
    if (err != cudaSuccess) return fail_cuda(detail, err);
    return SGEMM_OK;
}

sgemm_status_t sgemm_selftest_bounded_wait(int which, void *stream_ptr) {
    t_last_error[0] = '\0';
    if (which != 0 && which != 1) return fail(SGEMM_ERR_INVALID_VALUE, "which must be 0 or 1");
    if (!have_device()) return fail(SGEMM_ERR_UNSUPPORTED, "no CUDA device available");
    cudaError_t err = sg::simt_selftest_wait(which, static_cast<cudaStream_t>(stream_ptr));
    if (err != cudaSuccess) return fail_cuda("self-test kernel launch", err);
    return SGEMM_OK;
}

sgemm_status_t sgemm_fused_strided_batched(sgemm_op_t transa, sgemm_op_t transb,
                                           sgemm_path_t path, int64_t M, int64_t N, int64_t K,
                                           float alpha, const float *A, int64_t lda,
                                           int64_t strideA, const float *B, int64_t ldb,
                                           int64_t strideB, float beta, float *C, int64_t ldc,
                                           int64_t strideC, int64_t batch, const float *bias,
                                           sgemm_activation_t act, void *stream) {
    t_last_error[0] = '\0';
    if (act < SGEMM_ACT_NONE || act > SGEMM_ACT_SILU)
        return fail(SGEMM_ERR_INVALID_VALUE, "unknown activation");
    if ((transa != SGEMM_OP_N && transa != SGEMM_OP_T) ||
        (transb != SGEMM_OP_N && transb != SGEMM_OP_T))
        return fail(SGEMM_ERR_INVALID_VALUE, "transa and transb must be SGEMM_OP_N or SGEMM_OP_T");
    Path pth;
    switch (path) {
        case SGEMM_PATH_SIMT: pth = kPathSimt; break;
        case SGEMM_PATH_3XTF32: pth = kPathTf32x3; break;
        case SGEMM_PATH_TF32: pth = kPathTf32; break;
        default: return fail(SGEMM_ERR_INVALID_VALUE, "unknown path");
    }
    Args a{M, N, K, alpha, beta, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, batch};
    a.ta = transa == SGEMM_OP_T;
    a.tb = transb == SGEMM_OP_T;
    a.bias = bias;
    a.act = static_cast<int>(act);
    return dispatch(a, stream, pth);
}

sgemm_status_t sgemm_fused(sgemm_op_t transa, sgemm_op_t transb, sgemm_path_t path, int64_t M,
                           int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                           const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                           const float *bias, sgemm_activation_t act, void *stream) {
    return sgemm_fused_strided_batched(transa, transb, path, M, N, K, alpha, A, lda, 0, B, ldb, 0,
                                       beta, C, ldc, 0, 1, bias, act, stream);
}

sgemm_status_t sgemm_ex_strided_batched(sgemm_op_t transa, sgemm_op_t transb, sgemm_path_t path,
                                        int64_t M, int64_t N, int64_t K, float alpha,
                                        const float *A, int64_t lda, int64_t strideA,
                                        const float *B, int64_t ldb, int64_t strideB, float beta,
                                        float *C, int64_t ldc, int64_t strideC, int64_t batch,
                                        void *stream) {
    t_last_error[0] = '\0';
    if ((transa != SGEMM_OP_N && transa != SGEMM_OP_T) ||
        (transb != SGEMM_OP_N && transb != SGEMM_OP_T))
        return fail(SGEMM_ERR_INVALID_VALUE, "transa and transb must be SGEMM_OP_N or SGEMM_OP_T");
    Path pth;
    switch (path) {
        case SGEMM_PATH_SIMT: pth = kPathSimt; break;
        case SGEMM_PATH_3XTF32: pth = kPathTf32x3; break;
        case SGEMM_PATH_TF32: pth = kPathTf32; break;
        default: return fail(SGEMM_ERR_INVALID_VALUE, "unknown path");
    }
    Args a{M, N, K, alpha, beta, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, batch};
    a.ta = transa == SGEMM_OP_T;
    a.tb = transb == SGEMM_OP_T;
    return dispatch(a, stream, pth);
}

sgemm_status_t sgemm_ex(sgemm_op_t transa, sgemm_op_t transb, sgemm_path_t path, int64_t M,
                        int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                        const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                        void *stream) {
    return sgemm_ex_strided_batched(transa, transb, path, M, N, K, alpha, A, lda, 0, B, ldb, 0,
                                    beta, C, ldc, 0, 1, stream);
}

sgemm_status_t sgemm_host(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                          int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                          int64_t ldc, void *stream_ptr) {
    Args a{M, N, K, alpha, beta, A, lda, 0, B, ldb, 0, C, ldc, 0, 1};
    t_last_error[0] = '\0';
    sgemm_status_t st = validate(a);
    if (st != SGEMM_OK) return st;
    if (is_noop(a)) return SGEMM_OK;
    st = check_limits(a);
    if (st != SGEMM_OK) return st;
    if (!have_device()) return fail(SGEMM_ERR_UNSUPPORTED, "no CUDA device available");
    const sg::HostProblem hp{M, N, K, alpha, beta, A, lda, B, ldb, C, ldc};
    const char *detail = "";
    cudaError_t err = sg::host_gemm(hp, static_cast<cudaStream_t>(stream_ptr), chunk_gemm, &detail);
    if (err != cudaSuccess) {
        if (t_last_error[0] != '\0') return SGEMM_ERR_LAUNCH;  // the chunk's own message stands
        return fail_cuda(detail, err);
    }
    return SGEMM_OK;
}

const char *sgemm_status_string(sgemm_status_t status) {
    switch (status) {
        case SGEMM_OK: return "SGEMM_OK";
        case SGEMM_ERR_INVALID_VALUE: return "SGEMM_ERR_INVALID_VALUE";
        case SGEMM_ERR_LAUNCH: return "SGEMM_ERR_LAUNCH";
        case SGEMM_ERR_TIMEOUT: return "SGEMM_ERR_TIMEOUT";
        case SGEMM_ERR_UNSUPPORTED: return "SGEMM_ERR_UNSUPPORTED";
    }
    return "SGEMM_(unknown status)";
}

const char *sgemm_last_error(void) { return t_last_error; }

sgemm_status_t sgemm_device_status(void *stream_ptr) {
    t_last_error[0] = '\0';
    if (!have_device()) return fail(SGEMM_ERR_UNSUPPORTED, "no CUDA device available");
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    cudaError_t err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return fail_cuda("stream synchronize", err);
    const unsigned int word = sg::take_fault_words(stream);
    if (word & sg::kFaultTimeout)
        return fail(SGEMM_ERR_TIMEOUT, "a bounded wait inside a kernel expired");
    return SGEMM_OK;
}

sgemm_status_t sgemm_release_workspace(void) {
    t_last_error[0] = '\0';
    if (!have_device()) return SGEMM_OK;
    cudaError_t err = cudaDeviceSynchronize();
    if (err != cudaSuccess) return fail_cuda("device synchronize", err);
    err = sg::release_workspaces();
    cudaError_t err3 = sg::release_pack_workspaces();
    cudaError_t err4 = sg::release_host_buffers();
    if (err3 == cudaSuccess) err3 = err4;
    cudaError_t err2 = sg::tf32x3_release_workspaces();
    if (err == cudaSuccess) err = err3;
    if (err != cudaSuccess) return fail_cuda("workspace free", err);
    if (err2 != cudaSuccess) return fail_cuda("split workspace free", err2);
    return SGEMM_OK;
}

int sgemm_num_configs(void) { return sg::simt_num_configs(); }

const char *sgemm_config_name(int id) {
    if (id < 0 || id >= sg::simt_num_configs()) return nullptr;
    return sg::simt_config(id).name;
}

int sgemm_select_config(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                        int64_t lda, const float *B, int64_t ldb, const float *C, int64_t ldc,
                        int64_t batch) {
    Args a{M, N, K, alpha, 0.0f, A, lda, 0, B, ldb, 0, const_cast<float *>(C), ldc, 0, batch};
    if (batch > 1) {
        a.sA = M * lda;
        a.sB = K * ldb;
        a.sC = M * ldc;
    }
    if (validate(a) != SGEMM_OK || is_noop(a) || check_limits(a) != SGEMM_OK) return -1;
    if (alpha == 0.0f || K == 0) return -1;
    return choose_simt(to_problem(a));
}

sgemm_status_t sgemm_force_config(int id) {
    if (id < -1 || id >= sg::simt_num_configs())
        return fail(SGEMM_ERR_INVALID_VALUE, "unknown configuration id");
    g_forced_config.store(id);
    return SGEMM_OK;
}

}  // extern "C"
