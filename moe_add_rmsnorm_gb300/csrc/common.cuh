// Device helpers shared by the q8moe kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "q8moe.h"
#include "prefetch.h"

#define Q8_QBLOCK 32
#define Q8_WARPS 8          // warps per CTA in the streaming kernels
#define Q8_THREADS (Q8_WARPS * 32)

namespace q8 {

// ---- loads ------------------------------------------------------------------------------------------------------

// One 32-byte Q8_0 block of weights in one 256-bit load (sm_100+), read once: not kept in L1.
__device__ __forceinline__ void ld_block_stream(const int8_t* p, uint32_t (&w)[8]) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}

// Eight consecutive floats (32 bytes, 32-byte aligned) in one 256-bit load, read once: not kept in L1.
__device__ __forceinline__ void ld_f8_stream(const float* p, float* v) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
                 : "l"(p));
}

// A 32-byte block read through L1 (activations that several warps of the CTA share).
__device__ __forceinline__ void ld_block_shared_use(const int8_t* p, uint32_t (&w)[8]) {
    asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}

// A read-only f32 load whose issue order the compiler keeps relative to the other volatile loads: used for the few
// small values a kernel needs early, issued before its bulk weight loads so they do not queue behind them.
__device__ __forceinline__ float ld_f32_early(const float* p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_scale_stream(const float* p) {
    float v;
    asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// ---- int8 -> f32 --------------------------------------------------------------------------------------------------
// Byte i of w (a signed int8) as an exact f32: flip the sign bit to get b+128 in [0,255], place it in the low mantissa
// byte of 2^23 (0x4B000000), and subtract 2^23 + 128.  Both steps are exact.
template <int I>
__device__ __forceinline__ float i8_to_f32(uint32_t w_flipped) {
    return __uint_as_float(__byte_perm(w_flipped, 0x4B000000u, 0x7440u | I)) - 8388736.0f;
}

// ---- the per-block dot products --------------------------------------------------------------------------------

// f32 partial sum of one 32-value block: sum_t q[t] * x[t] (x in registers), four independent FMA chains.
__device__ __forceinline__ float block_dot_f32(const uint32_t (&w)[8], const float* __restrict__ x) {
    float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t u = w[i] ^ 0x80808080u;
        p0 = fmaf(i8_to_f32<0>(u), x[4 * i + 0], p0);
        p1 = fmaf(i8_to_f32<1>(u), x[4 * i + 1], p1);
        p2 = fmaf(i8_to_f32<2>(u), x[4 * i + 2], p2);
        p3 = fmaf(i8_to_f32<3>(u), x[4 * i + 3], p3);
    }
    return (p0 + p1) + (p2 + p3);
}

// Exact int32 dot of one weight block with one activation block (dp4a: four int8 products per instruction).
__device__ __forceinline__ int block_dot_i8(const uint32_t (&w)[8], const uint32_t (&x)[8]) {
    int d0 = 0, d1 = 0;
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        d0 = __dp4a((int)w[i], (int)x[i], d0);
        d1 = __dp4a((int)w[i + 1], (int)x[i + 1], d1);
    }
    return d0 + d1;
}

// ---- a lane's tile of weights and activation blocks -------------------------------------------------------------
// A lane owns BPL blocks (block indices bidx[j]) of RT consecutive rows.  The weights and scales of the whole tile are
// loaded before any of them is used, so RT*BPL 32-byte loads are in flight per lane.
template <int BPL, int RT>
struct WTile {
    uint32_t w[RT][BPL][8];
    float s[RT][BPL];
};

template <int BPL, int RT>
__device__ __forceinline__ void load_tile(WTile<BPL, RT>& t, const int8_t* __restrict__ q, const float* __restrict__ s,
                                          int64_t row0, int nvalid, int64_t k, int nb, const int (&bidx)[BPL],
                                          const bool (&bval)[BPL]) {
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
        for (int j = 0; j < BPL; ++j) {
            if (i < nvalid && bval[j]) {
                ld_block_stream(q + (row0 + i) * k + bidx[j] * 32, t.w[i][j]);
                t.s[i][j] = ld_scale_stream(s + (row0 + i) * nb + bidx[j]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) t.w[i][j][e] = 0u;
                t.s[i][j] = 0.f;
            }
        }
}

// The activation blocks a lane multiplies: f32 values (mode 0), int8 words and their scales (mode 1), or high and low
// words and their scales (mode 2).  The pointers may be global or shared memory.
template <int MODE, int BPL>
struct XTile {
    float f[MODE == 0 ? BPL : 1][MODE == 0 ? 32 : 1];
    uint32_t w[MODE >= 1 ? BPL : 1][8];
    uint32_t l[MODE == 2 ? BPL : 1][8];
    float s[BPL];
};

__device__ __forceinline__ void load_words32(const int8_t* p, uint32_t (&w)[8]) {
    const uint4 a = reinterpret_cast<const uint4*>(p)[0], b = reinterpret_cast<const uint4*>(p)[1];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

template <int MODE, int BPL>
__device__ __forceinline__ void load_x(XTile<MODE, BPL>& x, const float* xf, const int8_t* xq, const int8_t* xl,
                                       const float* xs, const int (&bidx)[BPL], const bool (&bval)[BPL]) {
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        if (MODE == 0) {
            const float4* p = reinterpret_cast<const float4*>(xf + bidx[j] * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 v = bval[j] ? p[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                x.f[j][4 * i + 0] = v.x;
                x.f[j][4 * i + 1] = v.y;
                x.f[j][4 * i + 2] = v.z;
                x.f[j][4 * i + 3] = v.w;
            }
            x.s[j] = 0.f;
        } else {
            if (bval[j]) {
                load_words32(xq + bidx[j] * 32, x.w[j]);
                if (MODE == 2) load_words32(xl + bidx[j] * 32, x.l[MODE == 2 ? j : 0]);
                x.s[j] = xs[bidx[j]];
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    x.w[j][e] = 0u;
                    x.l[MODE == 2 ? j : 0][e] = 0u;
                }
                x.s[j] = 0.f;
            }
        }
    }
}

template <int MODE>
struct AccType;
template <>
struct AccType<0> {
    using T = double;
};
template <>
struct AccType<1> {
    using T = float;
};
template <>
struct AccType<2> {
    using T = float;
};

// The two-word block dot: the exact integer 128 D(high words) + D(low words) (|.| < 2^27), which multiplies the block's
// scales and 1/128.
__device__ __forceinline__ int block_dot_i8x2(const uint32_t (&w)[8], const uint32_t (&xh)[8], const uint32_t (&xl)[8]) {
    return block_dot_i8(w, xh) * 128 + block_dot_i8(w, xl);
}

// This lane's share of row i of the tile: mode 0 adds each block's f32 partial, scaled, into f64; mode 1 scales each
// block's exact int32 dot by both block scales and adds in f32; mode 2 does the same with the two-word block dot and
// the scales times 1/128.
template <int MODE, int BPL, int RT>
__device__ __forceinline__ typename AccType<MODE>::T tile_row_dot(const WTile<BPL, RT>& t, int i,
                                                                  const XTile<MODE, BPL>& x) {
    typename AccType<MODE>::T acc = 0;
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        if (MODE == 0) {
            const float ps = block_dot_f32(t.w[i][j], x.f[j]);
            acc = fma((double)t.s[i][j], (double)ps, (double)acc);
        } else if (MODE == 1) {
            const int D = block_dot_i8(t.w[i][j], x.w[j]);
            acc = fmaf(t.s[i][j] * x.s[j], (float)D, (float)acc);
        } else {
            const int D = block_dot_i8x2(t.w[i][j], x.w[j], x.l[MODE == 2 ? j : 0]);
            acc = fmaf(t.s[i][j] * x.s[j] * 0.0078125f, (float)D, (float)acc);
        }
    }
    return acc;
}

// ---- reductions -----------------------------------------------------------------------------------------------

template <int LANES, typename T>
__device__ __forceinline__ T group_sum(T v) {
#pragma unroll
    for (int o = LANES / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---- the one-word activation quantizer ------------------------------------------------------------------------
// A warp holds one 32-value block, value `v` in lane `lane`.  d = amax / 127 and q = round-half-away(v / d), both
// divisions IEEE-rounded f32, q clamped to [-127, 127]; amax = 0 gives d = 0, q = 0.
//
// d: the product by fl32(1/127) corrected by one FMA residual step (Markstein's correction of a quotient by its exact
// remainder, P. Markstein, "Computation of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990), which equals the IEEE quotient for every non-negative finite float (checked exhaustively on the
// host over all 2,139,095,040 of them).
__device__ __forceinline__ float div127(float a) {
    const float c = 1.0f / 127.0f;
    const float q = __fmul_rn(a, c);
    return fmaf(fmaf(-q, 127.0f, a), c, q);
}

// The word needs only the integer the correctly rounded quotient rounds to.  The approximate quotient (__fdividef:
// within 2 ulp for a normal d, so within 2e-5 of v/d here, |v/d| <= 128) rounds to the same integer unless it lies
// within 1e-4 of a half-integer; there, and for a subnormal-range d, the IEEE quotient decides.
__device__ __forceinline__ bool quotient_near_tie(float t, float d) {
    const float a = fabsf(t);
    return d != 0.0f && (!(d >= 1e-30f) || fabsf((a - floorf(a)) - 0.5f) <= 1e-4f);
}

// N independent blocks at once (block i's value of this lane in v[i]): the N warp reductions interleaved, the
// quotients from reciprocals, and the IEEE division only on the rare warp that has a quotient near a half-integer.
template <int N>
__device__ __forceinline__ void quantize_lanes(const float (&v)[N], int8_t (&q)[N], float (&d)[N]) {
    float m[N], t[N];
#pragma unroll
    for (int i = 0; i < N; ++i) m[i] = fabsf(v[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int i = 0; i < N; ++i) m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], o));
    bool near = false;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        d[i] = div127(m[i]);
        t[i] = __fdividef(v[i], d[i]);
        near |= quotient_near_tie(t[i], d[i]);
    }
    if (__any_sync(0xffffffffu, near)) {  // warp-uniform, rare
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (quotient_near_tie(t[i], d[i])) t[i] = __fdiv_rn(v[i], d[i]);
    }
#pragma unroll
    for (int i = 0; i < N; ++i) q[i] = d[i] == 0.0f ? (int8_t)0 : (int8_t)(int)fminf(fmaxf(roundf(t[i]), -127.0f), 127.0f);
}

// The two-word form of N independent blocks (lane/mod.rs: the two-word activation): the one-word scale d and high word,
// and the low word = round-half-away(128 (t - hi)) of the IEEE quotient t = v / d itself (t - hi and the product by
// 128 are exact), so both words follow the correctly rounded quotient.
template <int N>
__device__ __forceinline__ void quantize2_lanes(const float (&v)[N], int8_t (&hi)[N], int8_t (&lo)[N], float (&d)[N]) {
    float m[N];
#pragma unroll
    for (int i = 0; i < N; ++i) m[i] = fabsf(v[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int i = 0; i < N; ++i) m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], o));
#pragma unroll
    for (int i = 0; i < N; ++i) {
        d[i] = div127(m[i]);
        if (d[i] == 0.0f) {
            hi[i] = 0;
            lo[i] = 0;
            continue;
        }
        const float t = __fdiv_rn(v[i], d[i]);
        const float r = fminf(fmaxf(roundf(t), -127.0f), 127.0f);
        const float f = fminf(fmaxf(roundf(__fmul_rn(__fsub_rn(t, r), 128.0f)), -127.0f), 127.0f);
        hi[i] = (int8_t)(int)r;
        lo[i] = (int8_t)(int)f;
    }
}

__device__ __forceinline__ int8_t quantize2_lane(float v, float& d_out, int8_t& lo_out) {
    const float vv[1] = {v};
    int8_t h[1], l[1];
    float d[1];
    quantize2_lanes<1>(vv, h, l, d);
    d_out = d[0];
    lo_out = l[0];
    return h[0];
}

__device__ __forceinline__ int8_t quantize_lane(float v, float& d_out) {
    const float vv[1] = {v};
    int8_t q[1];
    float d[1];
    quantize_lanes<1>(vv, q, d);
    d_out = d[0];
    return q[0];
}

// ---- pairs of f32 carrying about 44 significant bits ------------------------------------------------------------
// FP64 issues at a small fraction of the f32 rate on this part, so the few quantities that want more than 24 bits
// (a row's sum of squares, its norm factor, the product s * inv * w before its single rounding) are held as unevaluated
// sums hi + lo of two floats: Knuth's two-sum (TAOCP vol. 2, 4.2.2) and the FMA two-product are error-free
// transformations, and Dekker's normalisation (T. J. Dekker, "A floating-point technique for extending the available
// precision", Numer. Math. 18, 1971) keeps |lo| <= ulp(hi) / 2.
struct F2 {
    float hi, lo;
};

__device__ __forceinline__ F2 f2_quick(float a, float b) {  // |a| >= |b|
    const float s = a + b;
    return F2{s, b - (s - a)};
}

__device__ __forceinline__ F2 f2_two_sum(float a, float b) {
    const float s = a + b;
    const float bb = s - a;
    return F2{s, (a - (s - bb)) + (b - bb)};
}

__device__ __forceinline__ F2 f2_two_prod(float a, float b) {
    const float p = a * b;
    return F2{p, fmaf(a, b, -p)};
}

__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
    const F2 s = f2_two_sum(a.hi, b.hi);
    return f2_quick(s.hi, s.lo + (a.lo + b.lo));
}

// 1 / sqrt(m) for m > 0 given as a pair: the f32 reciprocal root refined by one Newton step whose residual
// 1 - m r^2 is formed with exact products (relative error of the pair about 2^-44).
__device__ __forceinline__ F2 f2_rsqrt(F2 m) {
    const float r = rsqrtf(m.hi);
    const F2 r2 = f2_two_prod(r, r);
    const F2 t = f2_two_prod(m.hi, r2.hi);
    // 1 - m r^2 = (1 - t.hi) - t.lo - m.hi r2.lo - m.lo r2.hi; 1 - t.hi is exact (t.hi is within a few ulp of 1)
    const float e = (((1.0f - t.hi) - t.lo) - m.hi * r2.lo) - m.lo * r2.hi;
    return f2_quick(r, r * (0.5f * e));
}

// f32(a * b * inv) with one rounding: a * b is an exact pair, multiplied by the pair inv to about 2^-44.
__device__ __forceinline__ float f2_mul3_round(float a, float b, F2 inv) {
    const F2 p = f2_two_prod(a, b);
    const F2 y = f2_two_prod(p.hi, inv.hi);
    const float lo = y.lo + fmaf(p.hi, inv.lo, p.lo * inv.hi);
    return y.hi + lo;
}

// ---- SiLU -------------------------------------------------------------------------------------------------------
// silu(z) = z / (1 + e^-z): for z << 0, e^-z overflows to +inf and the quotient is -0, the correct limit.
__device__ __forceinline__ float silu_f32(float z) { return __fdiv_rn(z, 1.0f + expf(-z)); }

// ---- grid-level arrival -----------------------------------------------------------------------------------------
// Release / acquire at GPU scope: orders this thread's earlier writes before its later ones as seen by other CTAs (and
// its later reads after what those CTAs released), without the sequentially consistent fence's cost.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// atomicAdd with acquire-release semantics at GPU scope: releases what this thread (and, through a preceding barrier,
// its CTA) wrote and acquires what earlier arrivals released, in one round trip.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* p, int v) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Called by every lane of a warp after the lanes' partial results are stored.  Returns true in every lane of the one
// warp that arrives last among `expected` arrivals on `counter`; that warp must reset the counter to 0 after reading
// the others' partials (through L2: __ldcg).
__device__ __forceinline__ bool warp_arrive_last(int* counter, int expected) {
    __syncwarp();  // orders the lanes' stores before lane 0's release (cumulative)
    int old = 0;
    if ((threadIdx.x & 31) == 0) old = atomic_add_acq_rel_gpu(counter, 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    const bool last = (old == expected - 1);
    __syncwarp();  // the other lanes read after lane 0's acquire
    return last;
}

// ---- L2 prefetch of weights the step reads later ----------------------------------------------------------------
// Bulk prefetch (TMA unit) of [p, p + n) into L2, in 64 KB pieces.  Only the 16-byte-aligned interior of a region is
// prefetched, so no piece reaches outside it.
constexpr unsigned long long kPrefetchPiece = 64ull << 10;

__device__ __forceinline__ void l2_prefetch_piece(const char* p, unsigned n) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(n) : "memory");
}

// Each (CTA, lane of warp 0) takes the pieces g = lane_index + m * (CTAs * 32) of the regions' concatenated pieces.
__device__ __forceinline__ void issue_l2_prefetch(const L2Prefetch& pf) {
    if (pf.n == 0 || threadIdx.x >= 32) return;
    const unsigned long long cta = blockIdx.x + (unsigned long long)gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    const unsigned long long step = (unsigned long long)gridDim.x * gridDim.y * gridDim.z * 32;
    const unsigned long long mine = cta * 32 + threadIdx.x;
    unsigned long long base = 0;  // global index of the region's first piece
    for (int r = 0; r < pf.n && r < L2Prefetch::kMax; ++r) {
        const uintptr_t a = ((uintptr_t)pf.ptr[r] + 15) & ~uintptr_t(15);
        const uintptr_t e = ((uintptr_t)pf.ptr[r] + pf.bytes[r]) & ~uintptr_t(15);
        if (e <= a) continue;
        const unsigned long long len = e - a;
        const unsigned long long np = (len + kPrefetchPiece - 1) / kPrefetchPiece;
        unsigned long long g = mine;
        if (g < base) g += (base - g + step - 1) / step * step;
        for (; g < base + np; g += step) {
            const unsigned long long off = (g - base) * kPrefetchPiece;
            const unsigned long long n = len - off < kPrefetchPiece ? len - off : kPrefetchPiece;
            l2_prefetch_piece((const char*)a + off, (unsigned)n);
        }
        base += np;
    }
}

// A cluster barrier split in two: arrive (releasing this thread's writes) now, wait (acquiring the others') later.
// Every thread of the CTA executes both, at warp-uniform points.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

}  // namespace q8
