// host_gemm.cu: C = alpha * (A . B) + beta * C with A, B and C in host memory.
//
// The rows of A (and of C when beta != 0) travel in chunks through two device buffers each,
// on an upload stream, while the caller's stream computes the previous chunk and a download
// stream returns the chunk before that. With page-locked host memory the copies overlap the
// GEMMs, so a long product runs at the slower of the copy rate and the kernel rate instead
// of their sum; with pageable memory everything runs in order on the caller's stream.
// B must be on the device before the first chunk can finish, so the first chunk is computed
// as K slices of growing size, each starting as soon as its rows of B and columns of A have
// arrived (later slices accumulate into C with beta = 1): the GPU starts after the first 256
// rows of B instead of all of them. Every GEMM is computed by the same device entry point (the SIMT path, with its
// per-shape configuration).
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "host_gemm.cuh"

namespace sg {
namespace {

struct HostPath {
    int dev = -1;
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t caller_done = nullptr;
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
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&h->caller_done, cudaEventDisableTiming);
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

// Copies `rows` rows of `width` bytes; one linear copy when both sides are contiguous.
cudaError_t copy_rows(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width,
                      size_t rows, cudaMemcpyKind kind, cudaStream_t stream) {
    if (dpitch == width && spitch == width)
        return cudaMemcpyAsync(dst, src, width * rows, kind, stream);
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, stream);
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

    // Chunks of whole 128-row tiles, at least an eighth of M, grown until one chunk holds half
    // a wave of 128 x 256 tiles (stream-K spreads such a chunk over every SM), at most M. At
    // 4096^3 from pinned memory (uploads run at about 200 GB/s): 1024-row chunks take 2.41 ms
    // per call, 2048-row chunks 2.46 ms, 512-row chunks 2.51 ms.
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        sms = 1;
    long long mc = (p.M + 7) / 8;
    mc = (mc + 127) / 128 * 128;
    if (mc < 128) mc = 128;
    const long long tiles_n = (p.N + 255) / 256;
    while (mc < p.M && 2 * (mc / 128) * tiles_n < sms) mc *= 2;
    if (mc > p.M) mc = p.M;
    // Device copies with rows padded to 16 bytes and buffers 256-byte aligned, so the
    // chunk GEMMs can always read them with TMA.
    const long long ldk = (p.K + 3) / 4 * 4, ldn = (p.N + 3) / 4 * 4;
    auto round64 = [](size_t n) { return (n + 63) / 64 * 64; };
    const size_t b_elems = round64(static_cast<size_t>(p.K) * ldn);
    const size_t a_elems = round64(static_cast<size_t>(mc) * ldk);
    const size_t c_elems = round64(static_cast<size_t>(mc) * ldn);
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

    // The first chunk in K slices that grow: the GPU starts once the first 256 rows of B (and
    // that slice of A) are up, and slice i is at most 256 + 0.4 x (the K already issued), so
    // each slice's upload (about 0.7 of its GEMM's time at 1024 x 4096 per k) lands before the
    // GEMMs ahead of it run out. Multiples of 32; a remainder under 128 joins the last slice.
    std::vector<long long> kslice = {0};
    if (reads_ab && p.K >= 512) {
        long long k = 0;
        while (k < p.K) {
            long long len = (256 + 2 * k / 5 + 31) / 32 * 32;
            if (p.K - (k + len) < 128) len = p.K - k;
            k += len;
            kslice.push_back(k);
        }
    } else {
        kslice.push_back(p.K);
    }
    const int kslices = static_cast<int>(kslice.size()) - 1;

    // The upload stream starts after everything already queued on the caller's stream.
    err = cudaEventRecord(h->caller_done, stream);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(up, h->caller_done, 0);
    if (err != cudaSuccess) {
        *detail = "ordering the upload stream failed";
        return err;
    }

    // Row chunks of mc rows; the last one (when it has at least 256 rows) in two halves, so
    // the download that ends the call is half as long.
    std::vector<long long> starts;
    for (long long r = 0; r < p.M; r += mc) starts.push_back(r);
    const long long last = starts.back(), last_rows = p.M - last;
    if (starts.size() > 1 && last_rows >= 256) starts.push_back(last + (last_rows / 2 + 127) / 128 * 128);
    starts.push_back(p.M);
    const long long chunks = static_cast<long long>(starts.size()) - 1;
    for (long long i = 0; i < chunks; ++i) {
        const int j = static_cast<int>(i & 1);
        const long long r0 = starts[i];
        const long long rows = starts[i + 1] - r0;
        // buffer j is free once chunk i - 2 has been downloaded
        if (i >= 2) err = cudaStreamWaitEvent(up, h->out_done[j], 0);
        if (err == cudaSuccess && reads_c)
            err = copy_rows(dC[j], ldn * sizeof(float), p.C + r0 * p.ldc,
                                    p.ldc * sizeof(float), p.N * sizeof(float), rows,
                                    cudaMemcpyHostToDevice, up);
        if (i == 0 && kslices > 1) {
            for (int si = 0; si < kslices && err == cudaSuccess; ++si) {
                const long long k0 = kslice[si], kn = kslice[si + 1] - kslice[si];
                err = copy_rows(dB + k0 * ldn, ldn * sizeof(float), p.B + k0 * p.ldb,
                                        p.ldb * sizeof(float), p.N * sizeof(float), kn,
                                        cudaMemcpyHostToDevice, up);
                if (err == cudaSuccess)
                    err = copy_rows(dA[0] + k0, ldk * sizeof(float), p.A + k0,
                                            p.lda * sizeof(float), kn * sizeof(float), rows,
                                            cudaMemcpyHostToDevice, up);
                if (err == cudaSuccess) err = cudaEventRecord(h->in_ready[0], up);
                if (err == cudaSuccess) err = cudaStreamWaitEvent(stream, h->in_ready[0], 0);
                if (err != cudaSuccess) {
                    *detail = "queuing a K slice's upload failed";
                    return err;
                }
                err = gemm(rows, p.N, kn, p.alpha, dA[0] + k0, ldk, dB + k0 * ldn, ldn,
                           k0 == 0 ? p.beta : 1.0f, dC[0], ldn, stream, detail);
                if (err != cudaSuccess) return err;
            }
        } else {
            if (i == 0 && err == cudaSuccess && reads_ab)
                err = copy_rows(dB, ldn * sizeof(float), p.B, p.ldb * sizeof(float),
                                        p.N * sizeof(float), p.K, cudaMemcpyHostToDevice, up);
            if (err == cudaSuccess && reads_ab)
                err = copy_rows(dA[j], ldk * sizeof(float), p.A + r0 * p.lda,
                                        p.lda * sizeof(float), p.K * sizeof(float), rows,
                                        cudaMemcpyHostToDevice, up);
            if (err == cudaSuccess) err = cudaEventRecord(h->in_ready[j], up);
            if (err == cudaSuccess) err = cudaStreamWaitEvent(stream, h->in_ready[j], 0);
            if (err != cudaSuccess) {
                *detail = "queuing a chunk's upload failed";
                return err;
            }
            err = gemm(rows, p.N, p.K, p.alpha, dA[j], ldk, dB, ldn, p.beta, dC[j], ldn, stream,
                       detail);
            if (err != cudaSuccess) return err;
        }
        err = cudaEventRecord(h->computed[j], stream);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(down, h->computed[j], 0);
        if (err == cudaSuccess)
            err = copy_rows(p.C + r0 * p.ldc, p.ldc * sizeof(float), dC[j],
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
