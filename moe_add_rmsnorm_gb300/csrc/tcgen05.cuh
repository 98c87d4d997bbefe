// 5th-generation tensor-core helpers (sm_100 family): shared-memory operand descriptors for the no-swizzle K-major
// layout, the f16 instruction descriptor, MMA issue and commit, and tensor-memory loads.
//
// Operand layout (no swizzle, K-major): an operand tile of R rows x K halves is cut into core matrices of 8 rows x 8
// halves (16 bytes a row, 128 bytes each); element (r, k) sits at (r / 8) * sbo + (k / 8) * 128 + (r % 8) * 16 +
// (k % 8) * 2, so the core matrices along K are 128 bytes apart (the leading byte offset) and the 8-row groups `sbo`
// bytes apart (the stride byte offset).
#pragma once
#include <stdint.h>

namespace q8 {

__device__ __forceinline__ uint32_t tc_smem(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Descriptor of a K-major no-swizzle operand starting at p (16-byte aligned), 8-row groups sbo bytes apart
// (descriptor version 1).
__device__ __forceinline__ uint64_t tc_desc(const void* p, uint32_t sbo) {
    return (uint64_t)((tc_smem(p) >> 4) & 0x3FFF) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) |
           (1ull << 46);
}

// kind::f16 instruction descriptor: D f32, A and B f16, both K-major, M x N.
__device__ __forceinline__ uint32_t tc_idesc_f16(int m, int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D[tmem] (+)= A * B^T for one K = 16 slice; acc 0 overwrites D.
__device__ __forceinline__ void tc_mma_f16(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{ .reg .pred p; setp.ne.u32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
                 ::"r"(tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// The MMAs issued so far by this thread arrive on bar when they complete.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(tc_smem(bar))
                 : "memory");
}

// 32 consecutive columns of this warp's 32 TMEM lanes (lane = thread), one 32-bit value each; complete after
// tc_wait_ld().
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace q8
