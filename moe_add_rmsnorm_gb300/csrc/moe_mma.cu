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
// its own; read-back warps take it with tcgen05.ld and add s_w * s_x * D into registers, the block order and the f32
// arithmetic of the int8 mode.  The CTA's warps split into three roles joined by mbarriers: fetch-and-convert (raw
// int8 tiles by cp.async four stages ahead, converted to f16 by a byte permute, exact, into one of two operand
// buffers), MMA issue (one thread, tcgen05.commit), and read-back (two TMEM buffers) — so conversion, tensor-core work
// and read-back of different stages overlap.  Operands use the no-swizzle K-major layout of 8-row x 16-byte core
// matrices.  One CTA per SM walks the items (group, 128-row tile, k slice) of the groups it takes; the k split is
// chosen per call from the number of such groups, and the last slice of a tile to finish adds the slices' partial sums
// in slice order.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "stream.cuh"

namespace q8 {
namespace {

constexpr int MM_M = 128;        // weight rows per tile: the MMA's M, one TMEM lane per thread
constexpr int MM_THREADS = 896;  // 28 warps in four roles (below)
constexpr int MM_NMAX = 64;      // group rows the kernel takes
constexpr int MM_MIN = 16;       // smaller groups stay on the CUDA cores
constexpr int MM_CORE = 128;     // bytes of one core matrix (8 rows x 16 bytes)
constexpr int MM_BPS = 2;        // 32-value blocks per pipeline stage (K = 64)
constexpr int MM_RING = 6;       // raw stages in the ring, filled by the tensor-copy producer
constexpr int MM_SMAX = 16;      // k slices per (group, tile) at most
constexpr int MM_SFOR = 130;     // eligible-group counts the host tabulates the k split for (the last for any more)
constexpr int MM_GCAP = 256;     // eligible groups listed in shared memory (beyond: found by a scan)
constexpr int MM_ROWB = MM_BPS * 32;                 // bytes of one raw row of a stage (int8)
constexpr int MM_KG = MM_BPS * 4;                    // f16 k-groups (core matrices) along K per stage
constexpr int MM_SBO = MM_KG * MM_CORE;              // bytes between row groups of an operand tile
constexpr int MM_SCB = 4;        // scale columns a tensor copy brings per row (16 bytes: the copy's minimum width)
// raw stage, as the tensor copies lay it out (every copy's destination 128-byte aligned): weights [mat][128][64 B]
// and weight scales [mat][128][4] (the 4-block column group holding the stage's 2 blocks)
constexpr int MM_RAW_W = 2 * MM_M * MM_ROWB;
constexpr int MM_RAW_SW = 2 * MM_M * MM_SCB * 4;
constexpr int MM_RAW = MM_RAW_W + MM_RAW_SW;
static_assert(MM_RAW % 128 == 0 && MM_RAW_W % 128 == 0, "tensor-copy destinations 128-byte aligned");
// operand buffer (f16, core-matrix layout): A per matrix [128 x 64], B [64 x 64]
constexpr int MM_OPA = MM_M * MM_ROWB * 2;
constexpr int MM_OPB = MM_NMAX * MM_ROWB * 2;
constexpr int MM_OP = 2 * MM_OPA + MM_OPB;
constexpr int MM_TCOLS = 512;    // TMEM: 2 buffers x 2 blocks x 2 matrices x 64 columns
constexpr int MM_SQ = 4;         // row-scale slots between the converters and the read-back
constexpr int MM_SCL = MM_BPS * MM_NMAX;  // floats of a slot: sx [2][64]
constexpr size_t MM_SMEM = (size_t)MM_RING * MM_RAW + 2 * MM_OP + (size_t)MM_SQ * MM_SCL * sizeof(float);
static_assert(MM_SMEM + 2048 <= 232448, "dynamic plus static shared memory within the 227 KB a CTA may hold");
constexpr int MM_CONV_WARPS = 10;                  // warps 0..9 convert
constexpr int MM_CONV_T = MM_CONV_WARPS * 32;
constexpr int MM_XT0 = MM_CONV_T - 4 * MM_NMAX;    // converter threads MM_XT0.. each own a quarter of a group row
constexpr int MM_WPT = 4;                          // weight row quarters a converter thread takes per stage, at most
constexpr int MM_XPD = 3;                          // stages the group-row loads run ahead of the conversion
static_assert(MM_XT0 >= 0 && MM_WPT * MM_CONV_T >= 2 * MM_M * 4, "converters cover a stage");
constexpr int MM_PROD_WARP = 10;                   // issues the tensor copies
constexpr int MM_ISSUE_WARP = 11;                  // lane 0 issues the MMAs
constexpr int MM_DRAIN_W0 = 12;                    // warps 12..27 read back: lanes 32*(w%4).., 16 columns each
constexpr int MM_DRAIN_WARPS = 16;
constexpr int MM_DCOLS = 16;                       // columns a read-back warp takes
constexpr int MM_DRAIN_T = MM_DRAIN_WARPS * 32;
static_assert(MM_DRAIN_W0 + MM_DRAIN_WARPS == MM_THREADS / 32, "roles cover the CTA");
static_assert(MM_DRAIN_W0 % 4 == 0 && MM_DRAIN_WARPS * MM_DCOLS == 4 * MM_NMAX, "read-back warps cover lanes and columns");

struct MmaParams {
    CUtensorMap tw0, tw1;  // weights [E*out_rows][k] int8, box 64 bytes x 128 rows (tw1: up, gate-up only)
    CUtensorMap ts0, ts1;  // weight scales [E*out_rows][nb] f32, box 4 x 128
    int gate_up;         // 1: gate and up (SiLU product to h); 0: down (per-choice outputs to part)
    int nmin;            // the fewest rows of a group this kernel takes (MM_MIN..MM_NMAX)
    int dense_rows;      // > 0: a dense projection: one group, matrix 0, rows 0 .. dense_rows - 1 (no plan lists)
    int E, out_rows, k, nb, K;
    const int32_t* offsets;
    const int32_t* lists;
    const int32_t* active;
    const int8_t* xq;    // gate-up: token rows [R][k] (choice c reads row c / K); down: hidden rows [R*K][k]
    const float* xs;
    float* out;          // gate-up: h [R*K][out_rows]; down: part [R*K][out_rows]
    const float* res;    // down only, or null: out = res + the product (same index; may alias out)
    int tiles;           // out_rows / 128
    int S;               // k slices per (group, tile) at most (scratch holds that many); 1: no split
    unsigned char s_for[MM_SFOR];  // the k slices to take for n eligible groups (n >= MM_SFOR - 1: the last)
    float* part;         // S > 1: [slots][tiles][S][2][64][128] scaled partial sums
    int* cnt;            // S > 1: [slots][tiles] arrivals (left zero)
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

// Two f32 lanes at once (sm_100+ packed f32 arithmetic; each lane rounds as the scalar instruction does).
__device__ __forceinline__ uint64_t pk2(float2 a) { return (uint64_t)__float_as_uint(a.x) | ((uint64_t)__float_as_uint(a.y) << 32); }
__device__ __forceinline__ float2 upk2(uint64_t r) {
    return make_float2(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32)));
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)));
    return upk2(r);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)), "l"(pk2(c)));
    return upk2(r);
}

// 16 bytes of read-only global memory (16-byte aligned).
__device__ __forceinline__ uint4 ldg_nc_v4(const int8_t* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// A tensor copy (TMA) of the 2-D tile at (x, y) into shared memory, counted on an mbarrier's transaction bytes.
__device__ __forceinline__ void tma_tile(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
                 : "memory");
}
// Four int8 (one 32-bit word) to four exact f16: 0x6400 | (v + 128) is the f16 1024 + v + 128, minus 1152.
__device__ __forceinline__ void i8x4_to_h(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const __half2 bias = __float2half2_rn(1152.0f);
    uint32_t a = __byte_perm(u, 0x64646464u, 0x7150), b = __byte_perm(u, 0x64646464u, 0x7352);
    __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias), hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
    lo = *reinterpret_cast<uint32_t*>(&ha);
    hi = *reinterpret_cast<uint32_t*>(&hb);
}

// 16 int8 (quarter q of a row of a stage) into f16 operand row r, k-groups 2q and 2q+1: row r lives in core
// row-group r/8, row r%8; its k-group g (values 8g..8g+7) at (r/8) * MM_SBO + g * 128 + (r%8) * 16.
__device__ __forceinline__ void convert_quarter(unsigned char* op, int r, int q, const uint4 v) {
    unsigned char* base = op + (size_t)(r >> 3) * MM_SBO + (r & 7) * 16 + 2 * q * MM_CORE;
    uint4 o0, o1;
    i8x4_to_h(v.x, o0.x, o0.y);
    i8x4_to_h(v.y, o0.z, o0.w);
    i8x4_to_h(v.z, o1.x, o1.y);
    i8x4_to_h(v.w, o1.z, o1.w);
    *reinterpret_cast<uint4*>(base) = o0;
    *reinterpret_cast<uint4*>(base + MM_CORE) = o1;
}

__device__ __forceinline__ void zero_quarter(unsigned char* op, int r, int q) {
    unsigned char* base = op + (size_t)(r >> 3) * MM_SBO + (r & 7) * 16 + 2 * q * MM_CORE;
    *reinterpret_cast<uint4*>(base) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(base + MM_CORE) = make_uint4(0, 0, 0, 0);
}

// Whether active group a is one this kernel takes (its expert id valid, MM_MIN..MM_NMAX rows).
__device__ __forceinline__ bool mm_eligible(const MmaParams& p, int a) {
    const int e = __ldg(p.active + 1 + a);
    if (e < 0 || e >= p.E) return false;
    const int n = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
    return n >= p.nmin && n <= MM_NMAX;
}

// Warp-wide scan of the active groups in order: returns how many are eligible; the first MM_GCAP go to list (when
// given) and the index of the target-th (0-based) to *found (when target >= 0 and it exists).
__device__ int mm_scan(const MmaParams& p, int nact, int* list, int target, int* found) {
    const int lane = threadIdx.x & 31;
    int count = 0;
    for (int a0 = 0; a0 < nact; a0 += 128) {
        bool el[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {  // four chunks' loads in flight
            const int a = a0 + 32 * u + lane;
            el[u] = a < nact && mm_eligible(p, a);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const unsigned bal = __ballot_sync(0xffffffffu, el[u]);
            const int pos = count + __popc(bal & ((1u << lane) - 1u));
            if (el[u] && list && pos < MM_GCAP) list[pos] = a0 + 32 * u + lane;
            if (el[u] && pos == target) *found = a0 + 32 * u + lane;
            count += __popc(bal);
        }
    }
    return count;
}

// The same for one thread alone: the index of the g-th eligible group by a serial scan (groups past the list only).
__device__ int mm_group_scan_one(const MmaParams& p, int nact, int g) {
    for (int a = 0, c = 0; a < nact; ++a)
        if (mm_eligible(p, a) && c++ == g) return a;
    return 0;
}

// A group: its expert (matrix) e, first choice c0 and rows n.
struct MmGroup {
    int e, c0, n;
};

// Choice i of a group starting at c0 (a dense projection's rows are its choices).
__device__ __forceinline__ int mm_choice(const MmaParams& p, int c0, int i) {
    return p.dense_rows ? i : __ldg(p.lists + c0 + i);
}

// The eligible group at position g of the order (warp-wide; the first MM_GCAP come from the list).
__device__ __forceinline__ int mm_group_at(const MmaParams& p, int nact, const int* glist, int g) {
    if (g < MM_GCAP) return glist[g];
    int found = 0;
    mm_scan(p, nact, nullptr, g, &found);
    return __reduce_max_sync(0xffffffffu, found);
}

// Group position g (warp-wide); a dense projection's one group needs no lookup.
__device__ __forceinline__ MmGroup mm_group(const MmaParams& p, int nact, const int* glist, int g) {
    if (p.dense_rows) return MmGroup{0, 0, p.dense_rows};
    const int e = __ldg(p.active + 1 + mm_group_at(p, nact, glist, g));
    const int c0 = __ldg(p.offsets + e);
    return MmGroup{e, c0, __ldg(p.offsets + e + 1) - c0};
}

// Persistent: the work is the items (eligible group g, tile, k slice) in that order, CTA b taking items b,
// b + gridDim.x, ...; an item covers weight rows tile*128 .. tile*128+127 of group g's expert against the group's n rows
// (16 <= n <= 64), k stages [slice*nst/S, (slice+1)*nst/S), S chosen per call from the number of eligible groups.
// Stage i covers blocks 2i, 2i+1.  The warps have four roles, handing stages on through mbarriers:
//  - warp 10 (the producer, one lane) brings each stage's weight tiles and their scales into one of MM_RING ring slots
//    with 2-D tensor copies; the slot's "full" barrier counts the bytes, and the slot is refilled once the converters
//    released it;
//  - warps 0..9 convert each raw stage to f16 operands (two buffers, each reused once the MMAs that read it completed),
//    together with the stage's slice of the group's rows, which they load from global memory a few stages ahead
//    (the rows are few and stay in L2), and copy the scales into one of MM_SQ scale slots (reused once the read-back
//    released it);
//  - warp 11 (one lane) issues the stage's MMAs, two per block and matrix (K = 16 each), into one of two TMEM buffers
//    (reused once the read-back released it) and commits them to the operand buffer's and the TMEM buffer's barriers;
//  - warps 12..27 read the TMEM buffer back (warp w: lanes 32*(w%4).., 16 columns), add s_w * s_x * D into registers
//    in block order, and after an item's last stage store its outputs (or its k slice's partial sums, the last slice
//    of a tile adding them in slice order).
// TMEM, buffers and barriers carry on from item to item: a running stage count gives slots, buffers and phases, so the
// roles run several stages apart.
__global__ void __launch_bounds__(MM_THREADS, 1) moe_mma_kernel(const __grid_constant__ MmaParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t raw_full[MM_RING], raw_empty[MM_RING];
    __shared__ __align__(8) uint64_t op_full[2], op_empty[2], tm_full[2], tm_empty[2], sc_full[MM_SQ], sc_empty[MM_SQ];
    __shared__ __align__(8) uint64_t tm_ready;  // the tensor memory is allocated
    __shared__ uint32_t tmem_base;
    __shared__ int choice_d[MM_NMAX];  // read-back: each group row's choice
    __shared__ int glist[MM_GCAP];     // the first eligible groups' indices in the active list
    __shared__ int nelig_s, a_d, last_d;
    const int t = threadIdx.x, w = t >> 5, lane = t & 31;
    griddep_wait();
    griddep_launch();
    const int nact = p.dense_rows ? 0 : __ldg(p.active);
    if (w == 0 && !p.dense_rows) {
        const int c = mm_scan(p, nact, glist, -1, nullptr);
        if (lane == 0) nelig_s = c;
    }
    __syncthreads();
    const int nelig = p.dense_rows ? 1 : nelig_s;
    const int nst_all = p.nb / MM_BPS;
    // k slices for this many eligible groups, chosen on the host (a loop of divisions here cost microseconds of
    // every launch's start)
    const int S = p.s_for[nelig < MM_SFOR ? nelig : MM_SFOR - 1];
    const int items = nelig * p.tiles * S;
    if ((int)blockIdx.x >= items) return;
    if (t == 0) {
        for (int i = 0; i < MM_RING; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], MM_CONV_WARPS + MM_DRAIN_WARPS);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&op_full[i], MM_CONV_WARPS);
            mbar_init(&op_empty[i], 1);
            mbar_init(&tm_full[i], 1);
            mbar_init(&tm_empty[i], MM_DRAIN_WARPS);
        }
        for (int i = 0; i < MM_SQ; ++i) {
            mbar_init(&sc_full[i], MM_CONV_WARPS);
            mbar_init(&sc_empty[i], MM_DRAIN_WARPS);
        }
        mbar_init(&tm_ready, 1);
        fence_barrier_init();
    }
    __syncthreads();
    // The tensor memory is allocated by the MMA-issue warp, which then releases the read-back warps through tm_ready;
    // the allocation takes microseconds, and the producer and the converters start their stages meanwhile.
    uint32_t tmem = 0;
    const int mats = p.gate_up ? 2 : 1;
    unsigned char* raw = smem;
    unsigned char* ops = smem + (size_t)MM_RING * MM_RAW;
    float* scl = reinterpret_cast<float*>(ops + 2 * (size_t)MM_OP);  // [MM_SQ] slots: sx [2][64]
    uint32_t gs = 0;  // stages this CTA has run (every role counts the same)
    bool ok = true;

    if (w == MM_PROD_WARP) {
        // ---- tensor-copy producer: weight tiles and their scales ---------------------------------------------------
        uint32_t issued = 0;  // stages whose copies were issued (the drain below waits for the last of them)
        if (lane == 0) {
            const unsigned bytes = (unsigned)(mats * (MM_M * MM_ROWB + MM_M * MM_SCB * 4));
            for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
                const int g = item / (p.tiles * S), tile = (item / S) % p.tiles, slice = item % S;
                const int a = p.dense_rows ? 0 : (g < MM_GCAP ? glist[g] : mm_group_scan_one(p, nact, g));
                const int e = p.dense_rows ? 0 : __ldg(p.active + 1 + a);
                const int wrow = e * p.out_rows + tile * MM_M;
                const int st0 = slice * nst_all / S, nst = (slice + 1) * nst_all / S - st0;
                for (int i = 0; i < nst && ok; ++i) {
                    const uint32_t gi = gs + i;
                    const int slot = gi % MM_RING;
                    if (gi >= MM_RING) ok = mbar_wait(&raw_empty[slot], ((gi / MM_RING) - 1) & 1, p.err);
                    if (!ok) break;
                    unsigned char* st = raw + (size_t)slot * MM_RAW;
                    const int b0 = (st0 + i) * MM_BPS;
                    mbar_arrive_expect_tx(&raw_full[slot], bytes);
                    tma_tile(st, &p.tw0, 32 * b0, wrow, &raw_full[slot]);
                    tma_tile(st + MM_RAW_W, &p.ts0, b0 & ~(MM_SCB - 1), wrow, &raw_full[slot]);
                    if (mats == 2) {
                        tma_tile(st + MM_M * MM_ROWB, &p.tw1, 32 * b0, wrow, &raw_full[slot]);
                        tma_tile(st + MM_RAW_W + MM_M * MM_SCB * 4, &p.ts1, b0 & ~(MM_SCB - 1), wrow, &raw_full[slot]);
                    }
                    ++issued;
                }
                gs += nst;
            }
            // every copy issued has landed before the CTA may end (bounded: a stalled pipeline already set the error)
            for (uint32_t gi = issued > MM_RING ? issued - MM_RING : 0; gi < issued; ++gi)
                mbar_wait(&raw_full[gi % MM_RING], (gi / MM_RING) & 1, p.err);
        }
        __syncwarp();
    } else if (w < MM_CONV_WARPS) {
        // ---- convert ----------------------------------------------------------------------------------------------
        // Per stage thread ct converts weight row quarters ct, ct + MM_CONV_T, ... from the raw stage, and threads
        // MM_XT0.. each one quarter (16 bytes) of a group row, loaded from global memory MM_XPD stages ahead into
        // registers; the threads holding quarter 0 of a row also load its two block scales.
        const int ct = t;  // 0 .. MM_CONV_T - 1
        const int xt = ct - MM_XT0, xr = xt >> 2, xqq = xt & 3;
        for (int item = blockIdx.x; item < items; item += gridDim.x) {
            const int g = item / (p.tiles * S), slice = item % S;
            const MmGroup grp = mm_group(p, nact, glist, g);
            const int c0 = grp.c0, n = grp.n;
            const int N = (n + 15) & ~15;
            const int st0 = slice * nst_all / S, nst = (slice + 1) * nst_all / S - st0;
            const bool xown = xt >= 0 && xr < n;  // this thread brings a real row quarter
            int64_t xrow = 0;
            if (xown) {
                const int c = mm_choice(p, c0, xr);
                xrow = p.gate_up ? c / p.K : c;
            }
            const int8_t* xsrc = p.xq + xrow * p.k + 16 * xqq;
            const float* ssrc = p.xs + xrow * p.nb;
            uint4 xb[MM_XPD];
            float2 sb[MM_XPD];
#pragma unroll
            for (int d = 0; d < MM_XPD; ++d) {
                xb[d] = make_uint4(0, 0, 0, 0);
                sb[d] = make_float2(0.f, 0.f);
                if (xown && d < nst) {
                    xb[d] = ldg_nc_v4(xsrc + 64 * (st0 + d));
                    if (xqq == 0) sb[d] = __ldg(reinterpret_cast<const float2*>(ssrc + MM_BPS * (st0 + d)));
                }
            }
            for (int i = 0; i < nst; ++i) {
                const uint32_t gi = gs + i;
                const int b = gi & 1, q = gi % MM_SQ, slot = gi % MM_RING;
                const uint4 xc = xb[0];
                const float2 sc = sb[0];
#pragma unroll
                for (int d = 0; d + 1 < MM_XPD; ++d) xb[d] = xb[d + 1], sb[d] = sb[d + 1];
                if (xown && i + MM_XPD < nst) {
                    xb[MM_XPD - 1] = ldg_nc_v4(xsrc + 64 * (st0 + i + MM_XPD));
                    if (xqq == 0) sb[MM_XPD - 1] = __ldg(reinterpret_cast<const float2*>(ssrc + MM_BPS * (st0 + i + MM_XPD)));
                }
                if (ok) ok = mbar_wait(&raw_full[slot], (gi / MM_RING) & 1, p.err);
                const unsigned char* st = raw + (size_t)slot * MM_RAW;
                if (ok && gi >= 2) ok = mbar_wait(&op_empty[b], ((gi >> 1) - 1) & 1, p.err);
                unsigned char* op = ops + (size_t)b * MM_OP;
                {  // weight row quarters: every load first, then the conversions
                    uint4 wv[MM_WPT];
#pragma unroll
                    for (int u = 0; u < MM_WPT; ++u) {
                        const int task = ct + u * MM_CONV_T;
                        if (task < mats * MM_M * 4) wv[u] = *reinterpret_cast<const uint4*>(st + (size_t)task * 16);
                    }
#pragma unroll
                    for (int u = 0; u < MM_WPT; ++u) {
                        const int task = ct + u * MM_CONV_T;
                        if (task < mats * MM_M * 4) {
                            const int row = task >> 2, m = row / MM_M;
                            convert_quarter(op + m * MM_OPA, row - m * MM_M, task & 3, wv[u]);
                        }
                    }
                }
                if (xown) convert_quarter(op + 2 * MM_OPA, xr, xqq, xc);
                else if (xt >= 0 && xr < N) zero_quarter(op + 2 * MM_OPA, xr, xqq);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the operands, to the tensor cores
                __syncwarp();
                if (lane == 0) mbar_arrive(&op_full[b]);
                if (ok && gi >= MM_SQ) ok = mbar_wait(&sc_empty[q], ((gi / MM_SQ) - 1) & 1, p.err);
                if (xt >= 0 && xqq == 0) {  // the stage's row scales into slot q (the weight scales stay in the raw slot)
                    float* sl = scl + (size_t)q * MM_SCL;
                    sl[xr] = sc.x;
                    sl[MM_NMAX + xr] = sc.y;
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&sc_full[q]);
                    mbar_arrive(&raw_empty[slot]);  // this warp is done with the raw stage
                }
            }
            gs += nst;
        }
    } else if (w == MM_ISSUE_WARP) {
        // ---- MMA issue --------------------------------------------------------------------------------------------
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                     "r"(MM_TCOLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        tmem = tmem_base;
        if (lane == 0) mbar_arrive(&tm_ready);
        for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
            const int g = item / (p.tiles * S), slice = item % S;
            const int n = mm_group(p, nact, glist, g).n;
            const int N = (n + 15) & ~15;
            const uint32_t idesc = mm_idesc(N);
            const int nst = (slice + 1) * nst_all / S - slice * nst_all / S;
            for (int i = 0; i < nst && ok; ++i) {
                const uint32_t gi = gs + i;
                const int b = gi & 1;
                if (lane == 0) {
                    if (ok) ok = mbar_wait(&op_full[b], (gi >> 1) & 1, p.err);
                    if (ok && gi >= 2) ok = mbar_wait(&tm_empty[b], ((gi >> 1) - 1) & 1, p.err);
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    if (ok) {
                        const unsigned char* op = ops + (size_t)b * MM_OP;
                        const uint32_t dbase = tmem + (uint32_t)(b * 256);
                        for (int j = 0; j < MM_BPS; ++j)
                            for (int m = 0; m < mats; ++m) {
                                const uint32_t d = dbase + j * 128 + m * 64;
                                const unsigned char* A = op + m * MM_OPA + j * 4 * MM_CORE;
                                const unsigned char* B = op + 2 * MM_OPA + j * 4 * MM_CORE;
                                mm_issue(d, mm_desc(A), mm_desc(B), idesc, 0u);                             // k 0..15
                                mm_issue(d, mm_desc(A + 2 * MM_CORE), mm_desc(B + 2 * MM_CORE), idesc, 1u);  // k 16..31
                            }
                        mm_commit(&op_empty[b]);
                        mm_commit(&tm_full[b]);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            }
            gs += nst;
        }
    } else {
        // ---- read-back, scaling and epilogue ----------------------------------------------------------------------
        const int dw = w - MM_DRAIN_W0;                 // 0 .. MM_DRAIN_WARPS - 1
        const int r = 32 * (w & 3) + lane;              // tile row = TMEM lane
        const int col0 = MM_DCOLS * (dw >> 2);          // this warp's columns
        const int dt = t - MM_DRAIN_W0 * 32;            // 0 .. MM_DRAIN_T - 1
        if (ok) ok = mbar_wait(&tm_ready, 0, p.err);    // the tensor memory is allocated
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        tmem = tmem_base;
        for (int item = blockIdx.x; item < items; item += gridDim.x) {  // (no early exit: named barriers below)
            const int g = item / (p.tiles * S), tile = (item / S) % p.tiles, slice = item % S;
            if (dw == 0 && !p.dense_rows) {
                const int a = mm_group_at(p, nact, glist, g);
                if (lane == 0) a_d = a;
            }
            asm volatile("bar.sync 2, %0;" ::"n"(MM_DRAIN_T));
            int c0 = 0, n = p.dense_rows;
            if (!p.dense_rows) {
                const int e = __ldg(p.active + 1 + a_d);
                c0 = __ldg(p.offsets + e);
                n = __ldg(p.offsets + e + 1) - c0;
            }
            if (dt < n) choice_d[dt] = mm_choice(p, c0, dt);
            asm volatile("bar.sync 2, %0;" ::"n"(MM_DRAIN_T));
            const int N = (n + 15) & ~15;
            const int st0 = slice * nst_all / S, nst = (slice + 1) * nst_all / S - st0;
            float acc0[MM_DCOLS], acc1[MM_DCOLS];
#pragma unroll
            for (int c = 0; c < MM_DCOLS; ++c) acc0[c] = acc1[c] = 0.f;
            const uint32_t lane_base = tmem + ((uint32_t)(32 * (w & 3)) << 16);
            for (int i = 0; i < nst; ++i) {
                const uint32_t gi = gs + i;
                const int b = gi & 1, q = gi % MM_SQ, slot = gi % MM_RING;
                const int jo = ((st0 + i) * MM_BPS) & (MM_SCB - 1);  // the stage's blocks inside the copied scale columns
                if (ok) ok = mbar_wait(&tm_full[b], (gi >> 1) & 1, p.err);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (ok) ok = mbar_wait(&sc_full[q], (gi / MM_SQ) & 1, p.err);
                if (ok) ok = mbar_wait(&raw_full[slot], (gi / MM_RING) & 1, p.err);  // (complete: the weight scales)
                const float* sl = scl + (size_t)q * MM_SCL;
                const float* swr = reinterpret_cast<const float*>(raw + (size_t)slot * MM_RAW + MM_RAW_W) + r * MM_SCB + jo;
                if (ok && col0 < N) {  // warp-uniform
#pragma unroll
                    for (int j = 0; j < MM_BPS; ++j) {
                        const float4* sxj = reinterpret_cast<const float4*>(sl + j * MM_NMAX + col0);
#pragma unroll
                        for (int m = 0; m < 2; ++m) {
                            if (m == 1 && !p.gate_up) break;
                            uint32_t v[16];
                            tmem_ld16(lane_base + (uint32_t)(b * 256 + j * 128 + m * 64 + col0), v);
                            // the scales load while the accumulator values travel
                            const float swv = swr[m * MM_M * MM_SCB + j];
                            float4 x4[4];  // the block's row scales for this warp's columns
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) x4[q4] = sxj[q4];
                            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                            float* acc = m == 0 ? acc0 : acc1;
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {  // s_w * s_x, then + (s_w * s_x) * D, two columns an instruction
                                const float2 s01 = mul2(make_float2(swv, swv), make_float2(x4[q4].x, x4[q4].y));
                                const float2 s23 = mul2(make_float2(swv, swv), make_float2(x4[q4].z, x4[q4].w));
                                float2 a01 = make_float2(acc[4 * q4], acc[4 * q4 + 1]);
                                float2 a23 = make_float2(acc[4 * q4 + 2], acc[4 * q4 + 3]);
                                a01 = fma2(s01, make_float2(__uint_as_float(v[4 * q4]), __uint_as_float(v[4 * q4 + 1])), a01);
                                a23 = fma2(s23, make_float2(__uint_as_float(v[4 * q4 + 2]), __uint_as_float(v[4 * q4 + 3])), a23);
                                acc[4 * q4] = a01.x;
                                acc[4 * q4 + 1] = a01.y;
                                acc[4 * q4 + 2] = a23.x;
                                acc[4 * q4 + 3] = a23.y;
                            }
                        }
                    }
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&tm_empty[b]);
                    mbar_arrive(&sc_empty[q]);
                    mbar_arrive(&raw_empty[slot]);
                }
            }
            gs += nst;
            const int orow = tile * MM_M + r;
            if (ok && S == 1) {
#pragma unroll
                for (int c = 0; c < MM_DCOLS; ++c) {
                    const int col = col0 + c;
                    if (col >= n) break;
                    const float v = p.gate_up ? silu_f32(acc0[c]) * acc1[c] : acc0[c];
                    const int64_t oi = (int64_t)choice_d[col] * p.out_rows + orow;
                    p.out[oi] = p.res ? p.res[oi] + v : v;
                }
            } else if (S > 1) {
                // K split: this slice's scaled sums to scratch; the last slice to arrive adds the slices in order
                // (every read-back thread passes the barriers, whatever its wait status)
                const int64_t pt = (int64_t)g * p.tiles + tile;
                const size_t slab = (size_t)2 * MM_NMAX * MM_M;
                float* mine = p.part + (size_t)(pt * S + slice) * slab;
                if (ok)
#pragma unroll
                    for (int c = 0; c < MM_DCOLS; ++c) {
                        const int col = col0 + c;
                        if (col >= n) break;
                        mine[(size_t)col * MM_M + r] = acc0[c];
                        if (p.gate_up) mine[(size_t)(MM_NMAX + col) * MM_M + r] = acc1[c];
                    }
                __threadfence();
                asm volatile("bar.sync 2, %0;" ::"n"(MM_DRAIN_T));
                if (dt == 0) last_d = atomic_add_acq_rel_gpu(p.cnt + pt, 1) == S - 1;
                asm volatile("bar.sync 2, %0;" ::"n"(MM_DRAIN_T));
                if (last_d && ok) {
                    const float* base = p.part + (size_t)(pt * S) * slab;
                    for (int c = 0; c < MM_DCOLS; ++c) {
                        const int col = col0 + c;
                        if (col >= n) break;
                        float gsum = 0.f, usum = 0.f;
                        for (int sl2 = 0; sl2 < S; ++sl2) {
                            gsum += __ldcg(base + (size_t)sl2 * slab + (size_t)col * MM_M + r);
                            if (p.gate_up) usum += __ldcg(base + (size_t)sl2 * slab + (size_t)(MM_NMAX + col) * MM_M + r);
                        }
                        const int64_t oi = (int64_t)choice_d[col] * p.out_rows + orow;
                        p.out[oi] = p.gate_up ? silu_f32(gsum) * usum : (p.res ? p.res[oi] + gsum : gsum);
                    }
                    if (dt == 0) p.cnt[pt] = 0;
                }
            }
            asm volatile("bar.sync 2, %0;" ::"n"(MM_DRAIN_T));  // choice_d and the flag are free for the next item
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (w == MM_ISSUE_WARP) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(MM_TCOLS));
}

}  // namespace

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The CUDA driver API's tensor-map encoder (cuTensorMapEncodeTiled), found once through the runtime's entry-point
// lookup, so the library does not link against libcuda.
EncodeTiled encode_tiled() {
    static const EncodeTiled fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeTiled) nullptr;
        return reinterpret_cast<EncodeTiled>(f);
    }();
    return fn;
}

// A 2-D row-major tensor [rows][cols] of u8 or f32 elements (row stride `stride` bytes) read in boxes of
// box_cols x box_rows; no swizzle, zero fill outside.
bool map_2d(CUtensorMap* m, bool f32, const void* base, uint64_t cols, uint64_t rows, uint64_t stride,
            uint32_t box_cols, uint32_t box_rows) {
    const EncodeTiled enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {stride};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base),
               dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool moe_mma_supported(const ExpertCall& c, bool dense) {
    // tensor copies: 16-byte aligned bases, row strides (k bytes, nb scales) multiples of 16 bytes, 4-column scale
    // boxes inside the rows, row coordinates that fit an int; a chunk's groups come from a plan
    return c.mode == 1 && (dense || c.plan.active) && c.R >= MM_MIN && c.out_rows % MM_M == 0 && c.k % (32 * MM_SCB) == 0 &&
           c.xq && c.xs && (uintptr_t)c.q0 % 16 == 0 && (!c.q1 || (uintptr_t)c.q1 % 16 == 0) &&
           (uintptr_t)c.xq % 16 == 0 && (uintptr_t)c.s0 % 16 == 0 && (!c.s1 || (uintptr_t)c.s1 % 16 == 0) &&
           (uintptr_t)c.xs % 16 == 0 && c.E * c.out_rows < ((int64_t)1 << 31) && c.R * c.K < ((int64_t)1 << 31) &&
           encode_tiled() != nullptr;
}

// The fewest rows of a group that takes the tensor cores (q8_set_grouped_tensor_core_rows); 0: none does.  Measured
// on correlated chunks (every group the chunk's rows): 16-row groups 89 us a chunk against 63 on the CUDA cores,
// 32-row groups 99 against 101, 64-row groups 99 against 176.
int kGroupedMmaMinRows = 32;

int moe_mma_min_rows() { return kGroupedMmaMinRows ? kGroupedMmaMinRows : MM_NMAX + 1; }

bool moe_mma_grouped(const ExpertCall& c) {
    return kGroupedMmaMinRows && c.R >= kGroupedMmaMinRows && moe_mma_supported(c);
}
int moe_mma_max_rows() { return MM_NMAX; }

cudaError_t launch_moe_mma(const ExpertCall& c, float* out, int max_groups, Carve& ws, cudaStream_t st,
                           const float* res, int nmin, int dense_rows) {
    if (!moe_mma_supported(c, dense_rows > 0)) return cudaErrorInvalidConfiguration;
    MmaParams p = {};
    // K split: up to MM_SMAX slices of at least 2 stages, as many as the workspace holds the partial sums of (the
    // kernel picks the number per call from the groups it finds; few groups, a dense projection's one, want many)
    const int nst_all = (int)(c.k / 32) / MM_BPS;
    int S = nst_all / 2;
    S = S < 1 ? 1 : (S > MM_SMAX ? MM_SMAX : S);
    const int tiles = (int)(c.out_rows / MM_M);
    if (nmin < MM_MIN || nmin > MM_NMAX) return cudaErrorInvalidValue;
    const int64_t slots = std::min<int64_t>(max_groups, c.R * c.K / nmin);  // eligible groups at most
    for (; S > 1; S = S > 4 ? S / 2 : S - 1) {
        const size_t bytes = (size_t)slots * tiles * S * 2 * MM_NMAX * MM_M * sizeof(float);
        const size_t at = (ws.used + 255) & ~size_t(255);
        if (at + bytes <= ws.size && ws.used_counters + (size_t)slots * tiles <= ws.n_counters) {
            p.part = ws.take<float>(bytes / sizeof(float));
            p.cnt = ws.take_counters((size_t)slots * tiles);
            break;
        }
    }
    const uint64_t nb = (uint64_t)(c.k / 32), wrows = (uint64_t)(c.E * c.out_rows);
    bool maps = map_2d(&p.tw0, false, c.q0, (uint64_t)c.k, wrows, (uint64_t)c.k, MM_ROWB, MM_M) &&
                map_2d(&p.ts0, true, c.s0, nb, wrows, nb * 4, MM_SCB, MM_M);
    if (maps && c.q1)
        maps = map_2d(&p.tw1, false, c.q1, (uint64_t)c.k, wrows, (uint64_t)c.k, MM_ROWB, MM_M) &&
               map_2d(&p.ts1, true, c.s1, nb, wrows, nb * 4, MM_SCB, MM_M);
    if (!maps) return cudaErrorInvalidValue;
    p.S = S;
    p.gate_up = c.q1 != nullptr;
    p.nmin = nmin;
    p.dense_rows = dense_rows;
    if (dense_rows && (c.E != 1 || c.K != 1 || c.R != dense_rows || dense_rows > MM_NMAX)) return cudaErrorInvalidValue;
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
    p.res = res;
    p.tiles = (int)(c.out_rows / MM_M);
    p.err = c.err;
    cudaError_t e = cudaFuncSetAttribute(moe_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)MM_SMEM);
    if (e != cudaSuccess) return e;
    int64_t grid = slots * p.tiles * p.S;  // persistent: one CTA per SM at most
    if (grid > device_info().sms) grid = device_info().sms;
    if (grid < 1) grid = 1;
    // for each possible number of eligible groups, the k slices giving the fewest rounds of items over the grid times
    // the stages per item (plus two for fill and epilogue)
    for (int n = 0; n < MM_SFOR; ++n) {
        int64_t best = -1;
        p.s_for[n] = 1;
        for (int sl = 1; sl <= p.S; ++sl) {
            const int64_t its = (int64_t)n * p.tiles * sl;
            const int64_t cost = ((its + grid - 1) / grid) * ((nst_all + sl - 1) / sl + 2);
            if (best < 0 || cost < best) best = cost, p.s_for[n] = (unsigned char)sl;
        }
    }
    return launch(moe_mma_kernel, dim3((unsigned)grid), dim3(MM_THREADS), MM_SMEM, st, c.pdl, p);
}

bool dense_mma_supported(const GemvCall& g) {
    if (g.mode != 1 || g.R < MM_MIN || g.R > MM_NMAX || g.dots || g.norm_a || g.k % (32 * MM_SCB)) return false;
    if ((uintptr_t)g.xq % 16 || (uintptr_t)g.xs % 16 || !encode_tiled()) return false;
    for (int i = 0; i < g.nseg; ++i)
        if (g.seg[i].n % MM_M || (uintptr_t)g.seg[i].q % 16 || (uintptr_t)g.seg[i].s % 16) return false;
    return true;
}

// A dense projection of 16..64 activation rows (a prefill chunk's q/k/v or O) on the tensor cores: the grouped
// product's kernel with one group holding every row (known to the kernel: no plan lists, no group scan), each
// segment's matrix as the group's expert, the residual (when given) added in its epilogue.
cudaError_t launch_dense_mma(const GemvCall& g, Carve& ws, cudaStream_t st) {
    if (!dense_mma_supported(g)) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < g.nseg && e == cudaSuccess; ++i) {
        ExpertCall c;
        c.mode = 1;
        c.q0 = g.seg[i].q;
        c.s0 = g.seg[i].s;
        c.E = 1;
        c.out_rows = g.seg[i].n;
        c.k = g.k;
        c.R = g.R;
        c.K = 1;
        c.xq = g.xq;
        c.xs = g.xs;
        c.err = g.err;
        c.pdl = g.pdl;
        Carve cv = ws;  // each segment's launch may reuse the same scratch after the one before it
        e = launch_moe_mma(c, g.seg[i].y, 1, cv, st, g.seg[i].residual, MM_MIN, (int)g.R);
    }
    return e;
}

}  // namespace q8
