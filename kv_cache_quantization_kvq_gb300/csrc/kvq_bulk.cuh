// kvq_bulk.cuh -- bulk asynchronous copies (global -> shared) completed on
// an mbarrier, for the staged quantize kernels (sm_90+ PTX, used on sm_103a).
//
// Every wait is bounded: after kWaitLimit polls the waiting thread records the
// failure in g_kvq_wait_timeouts and gives up instead of spinning forever.
#pragma once

#include <stdint.h>
#include <cuda.h>

namespace kvq {

// Count of bounded waits that gave up (never expected to be non-zero); one
// per translation unit that includes this header.
static __device__ unsigned int g_kvq_wait_timeouts;

// Host side: every translation unit that includes this header registers a
// reader of its own counter at load time; kvq_wait_timeouts() sums them.  A
// reader returns the error of the copy (its value is then not meaningful).
void register_wait_counter(cudaError_t (*read)(unsigned int*));

namespace {
cudaError_t read_wait_timeouts_of_this_unit(unsigned int* v)
{
    *v = 0u;
    return cudaMemcpyFromSymbol(v, g_kvq_wait_timeouts, sizeof *v);
}
const bool g_wait_counter_registered = (register_wait_counter(&read_wait_timeouts_of_this_unit), true);
}  // namespace

constexpr uint32_t kWaitLimit = 1u << 24;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make initialised barriers visible to the asynchronous (bulk copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// bytes (multiple of 16) from 16-byte aligned global memory into 16-byte
// aligned shared memory; completion is signalled on bar.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tiled tensor copy (TMA): the box at element coordinates (x, y) of the
// tensor described by map lands at smem_dst; completion counts the box bytes
// on bar.  x * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Prefetch bytes (multiple of 16) of 16-byte aligned global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

// One arrival (count 1) on bar, release semantics at CTA scope.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of bar to complete; false if the bound was hit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    atomicAdd(&g_kvq_wait_timeouts, 1u);
    return false;
}

}  // namespace kvq
