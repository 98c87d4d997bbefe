// A TMA-fed ring of shared-memory stages for streaming weight tiles (sm_90+ bulk copies, mbarrier completion).
//
// One producer thread issues `cp.async.bulk` copies of whole contiguous byte ranges (rows of quants, rows of scales)
// into stage s and arms stage s's "full" barrier with the byte count; consumer warps wait on "full", use the stage and
// arrive on its "empty" barrier; the producer waits on "empty" before refilling.  Every wait is bounded: after
// kWaitLimit polls the waiter records an error bit in the caller's error word and gives up, so a fault in the
// pipeline never hangs the GPU.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace q8 {

constexpr unsigned kWaitLimit = 1u << 22;  // polls (with back-off) before a wait gives up
constexpr int kErrPipeline = 4;            // error bit: a pipeline wait timed out

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete; false (and `err` |= kErrPipeline) after `limit` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, int* err, unsigned limit = kWaitLimit) {
    for (unsigned i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i > 64) __nanosleep(32);
    }
    if (err) atomicOr(err, kErrPipeline);
    return false;
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from global memory into shared memory,
// counted on `bar`'s transaction count.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

}  // namespace q8
