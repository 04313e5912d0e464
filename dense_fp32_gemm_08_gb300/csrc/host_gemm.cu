// host_gemm.cu: C = alpha * (A . B) + beta * C with A, B and C in host memory.
//
// B is uploaded once; the rows of A (and of C when beta != 0) then travel in chunks through
// two device buffers each, on an upload stream, while the caller's stream computes the
// previous chunk and a download stream returns the chunk before that. With page-locked host
// memory the copies overlap the GEMMs, so a long product runs at the slower of the copy rate
// and the kernel rate instead of their sum; with pageable memory everything runs in order on
// the caller's stream. Every chunk is computed by the same device
// entry point (the SIMT path, with its per-shape configuration).
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "host_gemm.cuh"

namespace sg {
namespace {

struct HostPath {
    int dev = -1;
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t b_ready = nullptr;
    cudaEvent_t in_ready[2] = {nullptr, nullptr};
    cudaEvent_t computed[2] = {nullptr, nullptr};
    cudaEvent_t out_done[2] = {nullptr, nullptr};
    float *buf = nullptr;  // B, then A[2], then C[2]
    size_t bytes = 0;
    std::mutex mu;         // one host-buffer product at a time per device
};

std::mutex g_host_mutex;
std::vector<HostPath *> g_host_paths;

cudaError_t host_path(int dev, HostPath **out) {
    std::lock_guard<std::mutex> lock(g_host_mutex);
    for (auto *h : g_host_paths)
        if (h->dev == dev) {
            *out = h;
            return cudaSuccess;
        }
    auto *h = new HostPath();
    h->dev = dev;
    cudaError_t err = cudaStreamCreateWithFlags(&h->up, cudaStreamNonBlocking);
    if (err == cudaSuccess) err = cudaStreamCreateWithFlags(&h->down, cudaStreamNonBlocking);
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&h->b_ready, cudaEventDisableTiming);
    for (int i = 0; i < 2 && err == cudaSuccess; ++i) {
        err = cudaEventCreateWithFlags(&h->in_ready[i], cudaEventDisableTiming);
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&h->computed[i], cudaEventDisableTiming);
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&h->out_done[i], cudaEventDisableTiming);
    }
    if (err != cudaSuccess) {
        delete h;
        return err;
    }
    g_host_paths.push_back(h);
    *out = h;
    return cudaSuccess;
}

// True when `ptr` is page-locked host memory (pinned or registered).
bool page_locked(const void *ptr) {
    if (!ptr) return true;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
        cudaGetLastError();  // clear the error of an unknown pointer
        return false;
    }
    return attr.type == cudaMemoryTypeHost;
}

}  // namespace

cudaError_t host_gemm(const HostProblem &p, cudaStream_t stream, DeviceGemmFn gemm,
                      const char **detail) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) {
        *detail = "cudaGetDevice failed";
        return err;
    }
    HostPath *h = nullptr;
    err = host_path(dev, &h);
    if (err != cudaSuccess) {
        *detail = "host-path streams / events could not be created";
        return err;
    }
    std::lock_guard<std::mutex> lock(h->mu);

    // Chunks of about an eighth of M, whole 128-row tiles, at least 128 rows.
    long long mc = (p.M + 7) / 8;
    mc = (mc + 127) / 128 * 128;
    if (mc < 128) mc = 128;
    if (mc > p.M) mc = p.M;
    const long long ldk = p.K, ldn = p.N;  // packed device copies
    const size_t b_elems = static_cast<size_t>(p.K) * ldn;
    const size_t a_elems = static_cast<size_t>(mc) * ldk;
    const size_t c_elems = static_cast<size_t>(mc) * ldn;
    const size_t need = (b_elems + 2 * a_elems + 2 * c_elems) * sizeof(float);
    if (h->bytes < need) {
        if (h->buf) {
            err = cudaFree(h->buf);
            h->buf = nullptr;
            h->bytes = 0;
            if (err != cudaSuccess) {
                *detail = "host-path buffer free failed";
                return err;
            }
        }
        err = cudaMalloc(&h->buf, need);
        if (err != cudaSuccess) {
            *detail = "host-path device buffers could not be allocated";
            return err;
        }
        h->bytes = need;
    }
    float *dB = h->buf;
    float *dA[2] = {dB + b_elems, dB + b_elems + a_elems};
    float *dC[2] = {dA[1] + a_elems, dA[1] + a_elems + c_elems};
    const bool reads_c = p.beta != 0.0f;
    const bool reads_ab = p.alpha != 0.0f && p.K > 0;
    // Copies from or to pageable memory are staged by the driver, and only their order within
    // one stream is guaranteed: with any pageable operand every copy and every chunk runs in
    // order on the caller's stream (no overlap); page-locked operands use the copy streams.
    const bool overlap = page_locked(p.C) && (!reads_ab || (page_locked(p.A) && page_locked(p.B)));
    cudaStream_t up = overlap ? h->up : stream;
    cudaStream_t down = overlap ? h->down : stream;

    // The upload stream starts after everything already queued on the caller's stream.
    err = cudaEventRecord(h->b_ready, stream);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(up, h->b_ready, 0);
    if (err == cudaSuccess && reads_ab)
        err = cudaMemcpy2DAsync(dB, ldn * sizeof(float), p.B, p.ldb * sizeof(float),
                                p.N * sizeof(float), p.K, cudaMemcpyHostToDevice, up);
    if (err == cudaSuccess) err = cudaEventRecord(h->b_ready, up);
    if (err != cudaSuccess) {
        *detail = "uploading B failed";
        return err;
    }

    const long long chunks = (p.M + mc - 1) / mc;
    for (long long i = 0; i < chunks; ++i) {
        const int j = static_cast<int>(i & 1);
        const long long r0 = i * mc;
        const long long rows = (p.M - r0) < mc ? (p.M - r0) : mc;
        // buffer j is free once chunk i - 2 has been downloaded
        if (i >= 2) err = cudaStreamWaitEvent(up, h->out_done[j], 0);
        if (err == cudaSuccess && reads_ab)
            err = cudaMemcpy2DAsync(dA[j], ldk * sizeof(float), p.A + r0 * p.lda,
                                    p.lda * sizeof(float), p.K * sizeof(float), rows,
                                    cudaMemcpyHostToDevice, up);
        if (err == cudaSuccess && reads_c)
            err = cudaMemcpy2DAsync(dC[j], ldn * sizeof(float), p.C + r0 * p.ldc,
                                    p.ldc * sizeof(float), p.N * sizeof(float), rows,
                                    cudaMemcpyHostToDevice, up);
        if (err == cudaSuccess) err = cudaEventRecord(h->in_ready[j], up);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(stream, h->in_ready[j], 0);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(stream, h->b_ready, 0);
        if (err != cudaSuccess) {
            *detail = "queuing a chunk's upload failed";
            return err;
        }
        err = gemm(rows, p.N, p.K, p.alpha, dA[j], ldk, dB, ldn, p.beta, dC[j], ldn, stream,
                   detail);
        if (err != cudaSuccess) return err;
        err = cudaEventRecord(h->computed[j], stream);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(down, h->computed[j], 0);
        if (err == cudaSuccess)
            err = cudaMemcpy2DAsync(p.C + r0 * p.ldc, p.ldc * sizeof(float), dC[j],
                                    ldn * sizeof(float), p.N * sizeof(float), rows,
                                    cudaMemcpyDeviceToHost, down);
        if (err == cudaSuccess) err = cudaEventRecord(h->out_done[j], down);
        if (err != cudaSuccess) {
            *detail = "queuing a chunk's download failed";
            return err;
        }
    }
    err = cudaStreamSynchronize(down);
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) *detail = "host-buffer product failed on the device";
    return err;
}

cudaError_t release_host_buffers() {
    std::lock_guard<std::mutex> lock(g_host_mutex);
    cudaError_t first = cudaSuccess;
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto *h : g_host_paths) {
        std::lock_guard<std::mutex> hl(h->mu);
        if (!h->buf) continue;
        cudaSetDevice(h->dev);
        cudaError_t err = cudaFree(h->buf);
        h->buf = nullptr;
        h->bytes = 0;
        if (err != cudaSuccess && first == cudaSuccess) first = err;
    }
    cudaSetDevice(cur);
    return first;
}

}  // namespace sg
