// ptx.cuh: thin inline-PTX wrappers for sm_103a (mbarrier, TMA, cp.async, bounded waits).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sg {

// Device error word: bit 0 = a bounded wait expired. Each translation unit that includes
// this header has its own copy (internal linkage, no relocatable device code needed) and
// registers a reader for it when the library loads; sgemm_device_status() reads and clears
// every registered word (take_fault_words).
static __device__ unsigned int g_fault_word;

// Host side of the fault words: the registry lives in sgemm_api.cu.
using FaultWordReader = unsigned int (*)(cudaStream_t);
void register_fault_word_reader(FaultWordReader reader);
// Reads and clears every translation unit's fault word on the current device (synchronising
// `stream`); returns their bitwise OR.
unsigned int take_fault_words(cudaStream_t stream);

namespace {
// Reads and clears this translation unit's fault word on the current device.
unsigned int take_unit_fault_word(cudaStream_t stream) {
    unsigned int word = 0;
    if (cudaMemcpyFromSymbolAsync(&word, g_fault_word, sizeof(word), 0, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess)
        return 0;
    const unsigned int zero = 0;
    cudaMemcpyToSymbolAsync(g_fault_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
    cudaStreamSynchronize(stream);
    return word;
}
[[maybe_unused]] const bool g_unit_fault_word_registered =
    (register_fault_word_reader(&take_unit_fault_word), true);
}  // namespace

constexpr unsigned int kFaultTimeout = 1u;
// Wall-clock limit of one bounded wait, in ns of %globaltimer. A legitimate wait inside these
// kernels lasts microseconds; the limit only ends a wait that can never complete.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void raise_fault(unsigned int bits) { atomicOr(&g_fault_word, bits); }

// ---- mbarrier --------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes initialised barriers visible to the async (TMA) proxy and to the other threads.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase with the given parity to complete. Returns false (and raises the
// device fault word) if it has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 63u) == 0u && globaltimer_ns() - t0 > kWaitLimitNs) {
            raise_fault(kFaultTimeout);
            return false;
        }
    }
}

// ---- TMA (cp.async.bulk.tensor), completion counted on an mbarrier ------------------------
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- cp.async (LDGSTS) with zero fill -------------------------------------------------------
// Copies `src_bytes` (0..4) bytes and zero-fills the rest of the 4-byte destination.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// Copies `src_bytes` (0..16) bytes and zero-fills the rest of the 16-byte destination.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace sg
