// Tensor-core products for a chunk's large expert groups: an expert chosen by at least 16 rows of the chunk has its
// weight tiles multiplied by all of those rows at once on the 5th-generation tensor cores.
//
// What it computes: the int8-activation projection of every row routed to the expert (lane/mod.rs module docs: one
// int8 word per value; the products by Q8_0 block, D[o,b] = sum over the block's 32 values of q_w * q_x as an exact
// integer, y[o] = sum_b s_w[o,b] * s_x[b] * D[o,b]) for the chunk's grouped expert products (lane_link.rs,
// Link::class_launch MoeTokenSort: a chunk's choices grouped by expert, each expert's weights read once; the pages'
// batch form multiplies the group with m16n8k32 int8 tensor tiles).
//
// How (GB300 design): the INT8 tensor rate of this part is far below its f16 rate, so the int8 quants and words are
// converted to f16 in shared memory — exactly: every |v| <= 127 is an f16 integer, every product is exact in the f32
// accumulator and so is every 32-value block sum (|D| <= 516,128 < 2^24).  For each 32-value block the tile's D
// (128 weight rows x N group rows) is formed by two tcgen05.mma kind::f16 (K = 16) into a tensor-memory accumulator of
// its own; the warpgroup reads it back with tcgen05.ld and adds s_w * s_x * D into registers, the block order and the
// f32 arithmetic of the int8 mode.  Raw int8 tiles stream into a ring of shared-memory stages by cp.async three
// stages ahead; each stage (two blocks) is converted to f16 by a byte permute (exact) into one of two operand buffers,
// and its MMAs run while the previous stage's accumulators (two TMEM buffers) are read back.  Operands use the
// no-swizzle K-major layout of 8-row x 16-byte core matrices.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "stream.cuh"

namespace q8 {
namespace {

constexpr int MM_M = 128;        // weight rows per tile: the MMA's M, one TMEM lane per thread
constexpr int MM_THREADS = 128;
constexpr int MM_NMAX = 64;      // group rows the kernel takes
constexpr int MM_MIN = 16;       // smaller groups stay on the CUDA cores
constexpr int MM_CORE = 128;     // bytes of one core matrix (8 rows x 16 bytes)
constexpr int MM_BPS = 2;        // 32-value blocks per pipeline stage (K = 64)
constexpr int MM_RING = 4;       // raw stages in flight (cp.async)
constexpr int MM_ROWB = MM_BPS * 32;                 // bytes of one raw row of a stage (int8)
constexpr int MM_KG = MM_BPS * 4;                    // f16 k-groups (core matrices) along K per stage
constexpr int MM_SBO = MM_KG * MM_CORE;              // bytes between row groups of an operand tile
// raw stage: weights [mat][128][64 B], activation rows [64][64 B], weight scales [mat][128][2], row scales [64][2]
constexpr int MM_RAW_W = 2 * MM_M * MM_ROWB;
constexpr int MM_RAW_X = MM_NMAX * MM_ROWB;
constexpr int MM_RAW_SW = 2 * MM_M * MM_BPS * 4;
constexpr int MM_RAW_SX = MM_NMAX * MM_BPS * 4;
constexpr int MM_RAW = MM_RAW_W + MM_RAW_X + MM_RAW_SW + MM_RAW_SX;
// operand buffer (f16, core-matrix layout): A per matrix [128 x 64], B [64 x 64]
constexpr int MM_OPA = MM_M * MM_ROWB * 2;
constexpr int MM_OPB = MM_NMAX * MM_ROWB * 2;
constexpr int MM_OP = 2 * MM_OPA + MM_OPB;
constexpr int MM_TCOLS = 512;    // TMEM: 2 buffers x 2 blocks x 2 matrices x 64 columns
constexpr size_t MM_SMEM = (size_t)MM_RING * MM_RAW + 2 * MM_OP;

struct MmaParams {
    int gate_up;         // 1: gate and up (SiLU product to h); 0: down (per-choice outputs to part)
    const int8_t* q0;    // gate (or down) [E*out_rows][k]
    const float* s0;
    const int8_t* q1;    // up
    const float* s1;
    int E, out_rows, k, nb, K;
    const int32_t* offsets;
    const int32_t* lists;
    const int32_t* active;
    const int8_t* xq;    // gate-up: token rows [R][k] (choice c reads row c / K); down: hidden rows [R*K][k]
    const float* xs;
    float* out;          // gate-up: h [R*K][out_rows]; down: part [R*K][out_rows]
    int tiles;           // out_rows / 128
    int* err;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// No-swizzle K-major descriptor: core matrices 128 B apart along K (leading byte offset), MM_SBO apart along M/N
// (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t mm_desc(const void* p) {
    return (uint64_t)((smem_u32(p) >> 4) & 0x3FFF) | ((uint64_t)(MM_CORE >> 4) << 16) | ((uint64_t)(MM_SBO >> 4) << 32) |
           (1ull << 46);
}

// kind::f16: D f32, A and B f16, both K-major, N and M.
__device__ __forceinline__ uint32_t mm_idesc(int n) { return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((MM_M >> 4) << 24); }

__device__ __forceinline__ void mm_issue(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{ .reg .pred p; setp.ne.u32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
                 ::"r"(tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mm_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
}

__device__ __forceinline__ void cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Four int8 (one 32-bit word) to four exact f16: 0x6400 | (v + 128) is the f16 1024 + v + 128, minus 1152.
__device__ __forceinline__ void i8x4_to_h(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const __half2 bias = __float2half2_rn(1152.0f);
    uint32_t a = __byte_perm(u, 0x64646464u, 0x7150), b = __byte_perm(u, 0x64646464u, 0x7352);
    __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias), hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
    lo = *reinterpret_cast<uint32_t*>(&ha);
    hi = *reinterpret_cast<uint32_t*>(&hb);
}

// One raw row of a stage (64 int8 = MM_BPS blocks) into f16 operand row r: row r lives in core row-group r/8, row
// r%8; its k-group g (values 8g..8g+7) at ((r/8) * MM_KG + g) * 128 + (r%8) * 16.
__device__ __forceinline__ void convert_row(unsigned char* op, int r, const unsigned char* raw) {
    unsigned char* base = op + (size_t)(r >> 3) * MM_SBO + (r & 7) * 16;
#pragma unroll
    for (int q = 0; q < MM_ROWB / 16; ++q) {  // 16 int8 = two k-groups
        const uint4 v = *reinterpret_cast<const uint4*>(raw + 16 * q);
        uint4 o0, o1;
        i8x4_to_h(v.x, o0.x, o0.y);
        i8x4_to_h(v.y, o0.z, o0.w);
        i8x4_to_h(v.z, o1.x, o1.y);
        i8x4_to_h(v.w, o1.z, o1.w);
        *reinterpret_cast<uint4*>(base + (2 * q) * MM_CORE) = o0;
        *reinterpret_cast<uint4*>(base + (2 * q + 1) * MM_CORE) = o1;
    }
}

__device__ __forceinline__ void zero_row(unsigned char* op, int r) {
    unsigned char* base = op + (size_t)(r >> 3) * MM_SBO + (r & 7) * 16;
#pragma unroll
    for (int g = 0; g < MM_KG; ++g) *reinterpret_cast<uint4*>(base + g * MM_CORE) = make_uint4(0, 0, 0, 0);
}

// CTA (group a, tile t): weight rows t*128 .. t*128+127 of the group's expert against the group's n rows (16 <= n <= 64).
// Stage i covers blocks 2i, 2i+1: its raw bytes arrive by cp.async up to MM_RING - 1 stages ahead (a ring slot is
// refilled once the stage it held has been read back, its scales included); the threads convert them
// to f16 operands (two buffers), thread 0 issues four MMAs per matrix (two per block, K = 16 each) into the stage's
// TMEM buffer, and stage i-1's accumulators are read back and scaled while stage i's MMAs run.
__global__ void __launch_bounds__(MM_THREADS, 1) moe_mma_kernel(const MmaParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar[2];
    __shared__ uint32_t tmem_base;
    __shared__ int rows_s[MM_NMAX];  // each group row's activation row
    __shared__ int choice_s[MM_NMAX];
    const int t = threadIdx.x, w = t >> 5;
    const int a = blockIdx.x / p.tiles, tile = blockIdx.x % p.tiles;
    griddep_wait();
    griddep_launch();
    if (a >= __ldg(p.active)) return;
    const int e = __ldg(p.active + 1 + a);
    if (e < 0 || e >= p.E) return;
    const int c0 = __ldg(p.offsets + e), n = __ldg(p.offsets + e + 1) - c0;
    if (n < MM_MIN || n > MM_NMAX) return;  // CTA-uniform: the CUDA-core kernel takes the group
    const int N = (n + 15) & ~15;
    if (t < n) {
        const int c = __ldg(p.lists + c0 + t);
        choice_s[t] = c;
        rows_s[t] = p.gate_up ? c / p.K : c;
    }
    if (t == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_barrier_init();
    }
    if (w == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                     "r"(MM_TCOLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base;
    const int mats = p.gate_up ? 2 : 1;
    const int64_t wrow = (int64_t)e * p.out_rows + (int64_t)tile * MM_M + t;  // this thread's weight row
    const int xrow = t < n ? rows_s[t] : 0;
    const uint32_t idesc = mm_idesc(N);
    const int nst = p.nb / MM_BPS;
    unsigned char* raw = smem;
    unsigned char* ops = smem + (size_t)MM_RING * MM_RAW;

    // this thread's share of raw stage i: its weight row(s) and scales, its group row and scales
    auto fetch = [&](int i) {
        unsigned char* st = raw + (size_t)(i % MM_RING) * MM_RAW;
        const int b0 = i * MM_BPS;
        for (int m = 0; m < mats; ++m) {
            const int8_t* q = (m == 0 ? p.q0 : p.q1) + wrow * p.k + 32 * b0;
            unsigned char* d = st + (size_t)(m * MM_M + t) * MM_ROWB;
#pragma unroll
            for (int u = 0; u < MM_ROWB / 16; ++u) cp16(d + 16 * u, q + 16 * u);
            cp8(st + MM_RAW_W + MM_RAW_X + (size_t)(m * MM_M + t) * MM_BPS * 4, (m == 0 ? p.s0 : p.s1) + wrow * p.nb + b0);
        }
        if (t < n) {
            const int8_t* x = p.xq + (int64_t)xrow * p.k + 32 * b0;
            unsigned char* d = st + MM_RAW_W + (size_t)t * MM_ROWB;
#pragma unroll
            for (int u = 0; u < MM_ROWB / 16; ++u) cp16(d + 16 * u, x + 16 * u);
            cp8(st + MM_RAW_W + MM_RAW_X + MM_RAW_SW + (size_t)t * MM_BPS * 4, p.xs + (int64_t)xrow * p.nb + b0);
        }
    };

    float acc0[MM_NMAX], acc1[MM_NMAX];
#pragma unroll
    for (int j = 0; j < MM_NMAX; ++j) acc0[j] = acc1[j] = 0.f;

    // stage i's accumulators (TMEM buffer i % 2: block j, matrix m at column (i%2)*256 + j*128 + m*64), scaled by the
    // raw stage's scales and added into acc in block order
    auto drain = [&](int i) {
        const unsigned char* st = raw + (size_t)(i % MM_RING) * MM_RAW;
        const float* sw = reinterpret_cast<const float*>(st + MM_RAW_W + MM_RAW_X);
        const float* sx = reinterpret_cast<const float*>(st + MM_RAW_W + MM_RAW_X + MM_RAW_SW);
        const uint32_t lane_base = tmem + ((uint32_t)(32 * w) << 16) + (uint32_t)((i & 1) * 256);
#pragma unroll
        for (int j = 0; j < MM_BPS; ++j)
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                if (m == 1 && !p.gate_up) break;
                const float swm = sw[(m * MM_M + t) * MM_BPS + j];
                // every 16-column load of the (block, matrix) accumulator issued, then one wait
                uint32_t r[MM_NMAX / 16][16];
#pragma unroll
                for (int c = 0; c < MM_NMAX / 16; ++c)
                    if (c * 16 < N) tmem_ld16(lane_base + j * 128 + m * 64 + c * 16, r[c]);  // CTA-uniform
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int c = 0; c < MM_NMAX / 16; ++c) {
                    if (c * 16 >= N) break;
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const float sc = swm * sx[(c * 16 + q) * MM_BPS + j];
                        if (m == 0) acc0[c * 16 + q] = fmaf(sc, __uint_as_float(r[c][q]), acc0[c * 16 + q]);
                        else acc1[c * 16 + q] = fmaf(sc, __uint_as_float(r[c][q]), acc1[c * 16 + q]);
                    }
                }
            }
    };

    for (int i = 0; i < MM_RING - 1; ++i) {  // the ring's first stages
        if (i < nst) fetch(i);
        cp_commit();
    }
    bool ok = true;
    for (int i = 0; i < nst; ++i) {
        cp_wait<MM_RING - 2>();  // raw stage i has landed (this thread's copies)
        __syncthreads();         // ... and every thread's
        // f16 operands of stage i in buffer i % 2 (its previous MMAs, stage i-2, completed before stage i-1 drained)
        {
            const unsigned char* st = raw + (size_t)(i % MM_RING) * MM_RAW;
            unsigned char* op = ops + (size_t)(i & 1) * MM_OP;
            for (int m = 0; m < mats; ++m) convert_row(op + m * MM_OPA, t, st + (size_t)(m * MM_M + t) * MM_ROWB);
            if (t < n) convert_row(op + 2 * MM_OPA, t, st + MM_RAW_W + (size_t)t * MM_ROWB);
            else if (t < N) zero_row(op + 2 * MM_OPA, t);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the operands, to the tensor cores
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (t == 0) {
            const unsigned char* op = ops + (size_t)(i & 1) * MM_OP;
            const uint32_t dbase = tmem + (uint32_t)((i & 1) * 256);
            for (int j = 0; j < MM_BPS; ++j)
                for (int m = 0; m < mats; ++m) {
                    const uint32_t d = dbase + j * 128 + m * 64;
                    const unsigned char* A = op + m * MM_OPA + j * 4 * MM_CORE;
                    const unsigned char* B = op + 2 * MM_OPA + j * 4 * MM_CORE;
                    mm_issue(d, mm_desc(A), mm_desc(B), idesc, 0u);  // k 0..15 of block j
                    mm_issue(d, mm_desc(A + 2 * MM_CORE), mm_desc(B + 2 * MM_CORE), idesc, 1u);  // k 16..31
                }
            mm_commit(&bar[i & 1]);
        }
        if (i > 0) {  // stage i-1 while stage i's MMAs run
            ok = mbar_wait(&bar[(i - 1) & 1], ((i - 1) >> 1) & 1, p.err) && ok;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (ok) drain(i - 1);
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        // the ring slot of stage i-1 (its scales were read by the drain above) takes stage i + MM_RING - 1
        if (ok && i + MM_RING - 1 < nst) fetch(i + MM_RING - 1);
        cp_commit();
        if (!ok) break;
    }
    cp_wait<0>();
    if (ok && nst > 0) {
        ok = mbar_wait(&bar[(nst - 1) & 1], ((nst - 1) >> 1) & 1, p.err);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (ok) drain(nst - 1);
    }
    if (ok) {
        const int orow = tile * MM_M + t;
#pragma unroll
        for (int j = 0; j < MM_NMAX; ++j) {
            if (j >= n) break;
            const float v = p.gate_up ? silu_f32(acc0[j]) * acc1[j] : acc0[j];
            p.out[(int64_t)choice_s[j] * p.out_rows + orow] = v;
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (w == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(MM_TCOLS));
}

}  // namespace

bool moe_mma_supported(const ExpertCall& c) {
    return c.mode == 1 && c.plan.active && c.R >= MM_MIN && c.out_rows % MM_M == 0 && c.k % (32 * MM_BPS) == 0 &&
           c.xq && c.xs && (uintptr_t)c.q0 % 16 == 0 && (!c.q1 || (uintptr_t)c.q1 % 16 == 0) &&
           (uintptr_t)c.xq % 16 == 0 && (uintptr_t)c.s0 % 8 == 0 && (!c.s1 || (uintptr_t)c.s1 % 8 == 0) &&
           (uintptr_t)c.xs % 8 == 0;
}

int moe_mma_min_rows() { return MM_MIN; }
int moe_mma_max_rows() { return MM_NMAX; }

cudaError_t launch_moe_mma(const ExpertCall& c, float* out, int max_groups, cudaStream_t st) {
    if (!moe_mma_supported(c)) return cudaErrorInvalidConfiguration;
    MmaParams p = {};
    p.gate_up = c.q1 != nullptr;
    p.q0 = c.q0;
    p.s0 = c.s0;
    p.q1 = c.q1;
    p.s1 = c.s1;
    p.E = (int)c.E;
    p.out_rows = (int)c.out_rows;
    p.k = (int)c.k;
    p.nb = (int)(c.k / 32);
    p.K = c.K;
    p.offsets = c.plan.offsets;
    p.lists = c.plan.lists;
    p.active = c.plan.active;
    p.xq = c.xq;
    p.xs = c.xs;
    p.out = out;
    p.tiles = (int)(c.out_rows / MM_M);
    p.err = c.err;
    cudaError_t e = cudaFuncSetAttribute(moe_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)MM_SMEM);
    if (e != cudaSuccess) return e;
    return launch(moe_mma_kernel, dim3((unsigned)(max_groups * p.tiles)), dim3(MM_THREADS), MM_SMEM, st, c.pdl, p);
}

}  // namespace q8
