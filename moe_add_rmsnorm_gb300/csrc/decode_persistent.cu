// The decode step's layers in one persistent launch: one CTA per SM, every CTA resident for the whole step, the
// dependent stages of a layer separated by grid-wide barriers instead of kernel boundaries.
//
// What it computes is the layer of the launch-per-stage path (qwen_emit docs, emit_qwen30b_generate: RMSNorm, q/k/v,
// per-head QK-norm + RoPE, attention over the cache, O with the residual, RMSNorm, softmax top-k router, SwiGLU
// experts, gated down-and-combine with the residual), in the int8 activation modes (lane/mod.rs: the one-word and the
// two-word activation), with the same block arithmetic: exact int32 block dots scaled by both block scales and summed
// in f32 per lane in block order, then across the warp.
//
// How (GB300 design): at one token a layer moves about 80 MB (64 MB of Q8_0 weights, 16.8 MB of cache at 4k
// positions), about 13 us at HBM speed, but each stage waits for the whole previous stage, and a launch per stage
// starts its weight stream only once its CTAs find room.  Here the weights and cache rows that do not depend on the
// token are copied into shared memory ahead of the stage that uses them by bulk copies (`cp.async.bulk`, completion
// counted on an mbarrier per region).  Issuing a bulk copy holds the issuing thread until the copy engine has taken
// most of its bytes, so one warp of the CTA (the producer) does nothing else; the other 11 (the compute warps) run the
// stages and tell the producer, through counters in shared memory, when a region is free again:
//   - q/k/v rows of layer l+1 as soon as O of layer l is done with the region, its router rows after the router,
//   - the cache rows of layer l+1 after the down-and-combine of layer l,
//   - O rows of layer l after its q/k/v projection,
//   - the chosen experts' down rows as soon as the routing is known,
// so that every stage but gate-up computes from shared memory as soon as its inputs from the other CTAs arrive.
// Gate-up streams its rows (about 180 KB a CTA) straight into registers, all requested at once.
//
// Stages (B = grid barrier):
//   A  every CTA norms the residual row and quantizes it; its share of the q/k/v rows      B
//   P  attention: CTA (g, j) takes positions [j c, (j+1) c) of key/value head g for the group's query heads; the
//      CTA holding the new position norms, turns and appends the new key and value rows; partial max, sum, values;
//      then the head's last CTAs to finish fold its partials, a (query head, 32-dim quarter) each, in partial order,
//      the output quantized per 32-value block                                                 B
//   O  its share of the O rows with the residual add                                          B
//   R  every CTA norms and quantizes the residual row; its share of the router rows           B
//   E  every CTA ranks the logits (top-k, renormalized gates); its share of the gate-up row pairs   B
//   D  every CTA quantizes the hidden rows; its share of the output rows of the chosen experts' down with the gated
//      combine and the residual add                                                          B (but the last layer)
//
// The grid barrier is one arrival counter that only grows within a launch (barrier k waits for (k+1) x CTAs
// arrivals); the last CTA out resets it.  Every wait is bounded: a grid wait that passes its cycle budget, an mbarrier
// wait that passes its poll limit or a producer wait that passes its budget records kErrPipeline in the error word and
// the CTA stops waiting for the rest of the launch (its results are then invalid and the step reports the error), so
// no fault hangs the GPU.  Co-residency of all CTAs is what cooperative launch guarantees (the launch fails rather than
// run part of the grid).
#include <float.h>

#include "common.cuh"
#include "kernels.h"
#include "stream.cuh"

namespace q8 {

int kPersistentDecode = 0;

namespace {

constexpr int PS_CW = 11;                // compute warps (12 warps a CTA: 3 per SM sub-partition, 168 registers)
constexpr int PS_CT = PS_CW * 32;        // compute threads
constexpr int PS_THREADS = PS_CT + 32;   // and the producer warp
constexpr int PS_HD = 128;               // head width
constexpr int PS_MAXG = 8;               // query heads per key/value head
constexpr int PS_MAXPPG = 64;            // attention CTAs per key/value head (partials a head folds)
constexpr int PS_MAXK = 32;              // kept experts
constexpr int PS_MAXE = 4096;            // experts ranked
constexpr int PS_MAXHHD = 4096;          // query heads x head width (the O projection's activation)
constexpr int PS_PVW = 8;                // warps whose value sums meet in shared memory (the rest fold into them)
constexpr long long kGridWaitCycles = 40000000ll;      // about 20 ms at 2 GHz
constexpr long long kProducerWaitCycles = 200000000ll; // about 100 ms: the producer may wait a whole layer

// ---- a CTA's shared memory ------------------------------------------------------------------------------------------

struct PsSmall {
    uint64_t bw, bc, br;           // fills of the W (q/k/v, then O), C (cache, then down) and R (router) regions
    int dead;                      // this CTA stopped waiting (a wait gave up)
    unsigned ev_w, ev_r, ev_route, ev_c;  // compute -> producer: regions free (counts that only grow)
    F2 nred[PS_CW + 1];            // norm: per-warp sums of squares, then the inverse root
    float stat[PS_MAXG][2];        // attention: the share's max and sum per head
    int kid[PS_MAXK];              // routing: kept experts in rank order, their logits and gates
    float kval[PS_MAXK];
    float gate[PS_MAXK];
    float den;                     // fold: the sum of weighted partial sums
    int ticket;                    // fold: this CTA's arrival rank among its key/value head's CTAs
};

inline size_t ps_align(size_t v) { return (v + 127) & ~size_t(127); }

// A pointer into the CTA's shared memory at byte offset `off`.  The offset passes through an opaque move, so the
// compiler forms the pointer where it is used instead of keeping every region's 64-bit address live across the
// whole layer loop (which would cost dozens of registers).
template <typename T>
__device__ __forceinline__ T* smp(unsigned char* sm, uint32_t off) {
    uint32_t o;
    asm volatile("mov.u32 %0, %1;" : "=r"(o) : "r"(off));
    return reinterpret_cast<T*>(sm + o);
}

// Offsets: the small state, the normed activation, a per-stage scratch union, then the three weight regions.  The
// attention's value sums meet in the C region's key rows when those are large enough (the keys are no longer needed
// then), else in the union.
PersistLayout ps_layout(const PersistDims& d, const PersistPlan& pl) {
    PersistLayout L{};
    const size_t two = d.mode == 2 ? 2 : 1;
    const size_t HHD = (size_t)d.H * PS_HD, KF = (size_t)d.K * d.F;
    const int G = d.KV > 0 ? d.H / d.KV : 1;
    size_t at = ps_align(sizeof(PsSmall));
    L.xq = (uint32_t)at;
    at = ps_align(at + d.D);
    L.xl = (uint32_t)at;
    at = ps_align(at + (two == 2 ? d.D : 0));
    L.xs = (uint32_t)at;
    at = ps_align(at + (size_t)d.D / 32 * 4);
    L.u = (uint32_t)at;
    const size_t red = (size_t)PS_PVW * G * PS_HD * 4;
    const bool red_in_c = (size_t)pl.capr * PS_HD * 4 >= red;
    // attention scratch
    size_t b = 0;
    L.b_qs = (uint32_t)b;
    b = ps_align(b + (size_t)G * PS_HD * 4);
    L.b_kn = (uint32_t)b;
    b = ps_align(b + PS_HD * 4);
    L.b_vn = (uint32_t)b;
    b = ps_align(b + PS_HD * 4);
    L.b_sc = (uint32_t)b;
    b = ps_align(b + (size_t)pl.capr * PS_MAXG * 4);
    L.b_red = red_in_c ? 0u : (uint32_t)b;  // relative to u, or (red_in_c) to the C region
    b = ps_align(b + (red_in_c ? 0 : red));
    // fold scratch
    size_t f = 0;
    L.f_red = (uint32_t)f;
    f = ps_align(f + (size_t)PS_CW * 32 * 4);
    // O scratch
    size_t o = 0;
    L.o_q = (uint32_t)o;
    o = ps_align(o + HHD);
    L.o_l = (uint32_t)o;
    o = ps_align(o + (two == 2 ? HHD : 0));
    L.o_s = (uint32_t)o;
    o = ps_align(o + HHD / 32 * 4);
    // routing scratch
    size_t e = 0;
    const size_t E8 = ((size_t)d.E + 7) & ~size_t(7);
    L.e_key = (uint32_t)e;
    e = ps_align(e + E8 * 4);
    L.e_val = (uint32_t)e;
    e = ps_align(e + E8 * 4);
    // down scratch
    size_t h = 0;
    L.d_q = (uint32_t)h;
    h = ps_align(h + KF);
    L.d_l = (uint32_t)h;
    h = ps_align(h + (two == 2 ? KF : 0));
    L.d_s = (uint32_t)h;
    h = ps_align(h + KF / 32 * 4);

    size_t um = b;
    if (f > um) um = f;
    if (o > um) um = o;
    if (e > um) um = e;
    if (h > um) um = h;
    at = ps_align(at + um);
    // weight regions
    const size_t wq = (size_t)pl.rq * (d.D + d.D / 8), wo = (size_t)pl.ro * (HHD + HHD / 8);
    L.w = (uint32_t)at;
    at = ps_align(at + (wq > wo ? wq : wo));
    const size_t cc = (size_t)pl.capr * 2 * PS_HD * 4, cd = (size_t)pl.rd * d.K * (d.F + d.F / 8);
    L.c = (uint32_t)at;
    at = ps_align(at + (cc > cd ? cc : cd));
    L.r = (uint32_t)at;
    at = ps_align(at + (size_t)pl.rr * (d.D + d.D / 8));
    L.total = (uint32_t)at;
    L.red_in_c = red_in_c ? 1u : 0u;
    return L;
}

// ---- synchronization ------------------------------------------------------------------------------------------------

// The compute warps' CTA barrier (the producer warp runs on its own).
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(PS_CT) : "memory"); }

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned atom_add_acq_rel_u32(unsigned* p, unsigned v) {
    unsigned o;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(o) : "l"(p), "r"(v) : "memory");
    return o;
}

__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// The grid barrier's arrival counter and, a line after it, the exit counter.  (Arrivals spread over eight counters on
// lines of their own, summed by each waiter, measured slower: the waiters' eight loads a poll cost more than the
// atomics' queueing on one line.)
constexpr int PS_BARS = 1;
constexpr int PS_GROUP_BAR = 128;  // unsigned ints: the attention's per-head arrival counters start 512 bytes in
constexpr int PS_MAXKV = 12;       // key/value heads with a counter of their own
constexpr int PS_BAR_STRIDE = 32;  // unsigned ints: 128 bytes
static_assert((PS_BARS + 1) * PS_BAR_STRIDE <= PS_GROUP_BAR, "barrier counters");
static_assert((PS_GROUP_BAR + PS_MAXKV * PS_BAR_STRIDE) * 4 <= kPersistBarBytes, "barrier counters");

__device__ __forceinline__ unsigned grid_arrivals(const unsigned* bar) {
    unsigned v[PS_BARS];
#pragma unroll
    for (int i = 0; i < PS_BARS; ++i) v[i] = ld_acquire_gpu(bar + i * PS_BAR_STRIDE);
    unsigned n = 0;
#pragma unroll
    for (int i = 0; i < PS_BARS; ++i) n += v[i];
    return n;
}

// Barrier k of the launch, for the compute warps: thread 0 arrives (releasing the CTA's writes, ordered before it by
// the CTA barrier) and waits for (k + 1) x CTAs arrivals (acquiring the others').
__device__ __forceinline__ void grid_barrier(unsigned* bar, unsigned k, int* err, PsSmall& s) {
    cbar();
    if (threadIdx.x == 0 && !s.dead) {
        const unsigned target = (k + 1) * gridDim.x;
        atom_add_acq_rel_u32(bar, 1u);
        const long long t0 = clock64();
        while ((int)(grid_arrivals(bar) - target) < 0) {
            if (clock64() - t0 > kGridWaitCycles || (*(volatile int*)err & kErrPipeline)) {
                atomicOr(err, kErrPipeline);
                s.dead = 1;
                break;
            }
        }
    }
    cbar();
}

// A region's fill: bounded wait (every compute thread) on its barrier's phase `n`, which then counts as completed.
// After a wait that gave up the CTA waits for nothing more; `n` stays uniform because every thread reads the flag after
// the CTA barrier.
__device__ __forceinline__ void region_wait(uint64_t* bar, unsigned& n, int* err, PsSmall& s) {
    if (!s.dead && !mbar_wait(bar, n & 1, err)) s.dead = 1;
    cbar();
    if (!s.dead) ++n;
}

// Compute warps -> producer: the region an event names is free (its count reached v).  Called after a CTA barrier.
__device__ __forceinline__ void signal(unsigned* ev, unsigned v) {
    if (threadIdx.x == 0) {
        __threadfence_block();
        *(volatile unsigned*)ev = v;
    }
}

// Producer: waits until the event's count reaches v; false after the budget (the CTA is then marked dead).
__device__ __forceinline__ bool producer_wait(const unsigned* ev, unsigned v, int* err, PsSmall& s) {
    const long long t0 = clock64();
    while ((int)(*(volatile const unsigned*)ev - v) < 0) {
        if (*(volatile int*)&s.dead) return false;
        if (clock64() - t0 > kProducerWaitCycles) {
            atomicOr(err, kErrPipeline);
            s.dead = 1;
            return false;
        }
        __nanosleep(64);
    }
    __threadfence_block();
    fence_proxy_async_smem();  // the compute warps' reads of the region come before the copies that overwrite it
    return true;
}

// ---- the fills (the producer issues them; the bytes of a fill are counted on its region's barrier) -----------------

// Rows [lo, hi) of one matrix (k columns, k/32 scales a row) into a region holding `cap` rows: quants of row r at
// (r - r0) * k, scales after all quants at cap * k + (r - r0) * (k / 8).
__device__ __forceinline__ void fill_rows(unsigned char* dst, int r0, int cap, const int8_t* q, const float* sc, int64_t q0,
                                          int lo, int hi, int k, uint64_t* bar) {
    if (hi <= lo) return;
    const unsigned n = (unsigned)(hi - lo);
    bulk_g2s(dst + (size_t)(lo - r0) * k, q + (q0 + lo) * k, n * (unsigned)k, bar);
    bulk_g2s(dst + (size_t)cap * k + (size_t)(lo - r0) * (k / 8), sc + (q0 + lo) * (k / 32), n * (unsigned)(k / 8), bar);
}

// This CTA's q/k/v rows [r0, r1) of the concatenation [q; k; v].
__device__ __noinline__ void fill_qkv(const PersistCall& p, const PersistLayer& ly, unsigned char* W, uint64_t* bar) {
    const PersistDims& d = p.dims;
    const int NQ = d.H * PS_HD, NK = d.KV * PS_HD, NR = NQ + 2 * NK;
    const int r0 = min((int)blockIdx.x * p.plan.rq, NR), r1 = min(r0 + p.plan.rq, NR);
    mbar_arrive_expect_tx(bar, (unsigned)(r1 - r0) * (unsigned)(d.D + d.D / 8));
    const int s0[3] = {0, NQ, NQ + NK}, s1[3] = {NQ, NQ + NK, NR};
    const int8_t* q[3] = {ly.wq_q, ly.wk_q, ly.wv_q};
    const float* sc[3] = {ly.wq_s, ly.wk_s, ly.wv_s};
    for (int i = 0; i < 3; ++i) {
        const int lo = max(r0, s0[i]), hi = min(r1, s1[i]);
        // rows of segment i are numbered from its start: shift so that fill_rows' row index is the global one
        fill_rows(W, r0, p.plan.rq, q[i], sc[i], -(int64_t)s0[i], lo, hi, d.D, bar);
    }
}

// This CTA's O rows.
__device__ __noinline__ void fill_o(const PersistCall& p, const PersistLayer& ly, unsigned char* W, uint64_t* bar) {
    const PersistDims& d = p.dims;
    const int HHD = d.H * PS_HD;
    const int r0 = min((int)blockIdx.x * p.plan.ro, d.D), r1 = min(r0 + p.plan.ro, d.D);
    mbar_arrive_expect_tx(bar, (unsigned)(r1 - r0) * (unsigned)(HHD + HHD / 8));
    fill_rows(W, r0, p.plan.ro, ly.wo_q, ly.wo_s, 0, r0, r1, HHD, bar);
}

// This CTA's router rows.
__device__ __noinline__ void fill_router(const PersistCall& p, const PersistLayer& ly, unsigned char* R, uint64_t* bar) {
    const PersistDims& d = p.dims;
    const int r0 = min((int)blockIdx.x * p.plan.rr, d.E), r1 = min(r0 + p.plan.rr, d.E);
    mbar_arrive_expect_tx(bar, (unsigned)(r1 - r0) * (unsigned)(d.D + d.D / 8));
    fill_rows(R, r0, p.plan.rr, ly.wr_q, ly.wr_s, 0, r0, r1, d.D, bar);
}

// The attention CTA's share of positions at cache length len: key/value head g = CTA / ppg, positions
// [p0, p0 + np) with p0 = (CTA % ppg) * chunk, chunk = ceil(len / ppg).  CTAs past the last head get none.
__device__ __forceinline__ void attn_share(const PersistCall& p, int len, int& g, int& p0, int& np) {
    g = (int)blockIdx.x / p.plan.ppg;
    const int j = (int)blockIdx.x % p.plan.ppg;
    const int chunk = (len + p.plan.ppg - 1) / p.plan.ppg;
    p0 = j * chunk;
    np = (g < p.dims.KV && len >= 1 && len <= p.dims.ctx) ? max(0, min(chunk, len - p0)) : 0;
}

// The cached key and value rows of this CTA's positions but the new one (len - 1, written during the step): keys at
// C, values capr rows later.
__device__ __noinline__ void fill_cache(const PersistCall& p, const PersistLayer& ly, int len, unsigned char* C, uint64_t* bar) {
    int g, p0, np;
    attn_share(p, len, g, p0, np);
    const int nold = (np > 0 && p0 + np == len) ? np - 1 : np;  // the new position is the share's last
    const unsigned row = PS_HD * 4;
    mbar_arrive_expect_tx(bar, 2u * (unsigned)nold * row);
    if (nold > 0) {
        const int64_t off = ((int64_t)g * p.dims.ctx + p0) * PS_HD;
        bulk_g2s(C, ly.kc + off, (unsigned)nold * row, bar);
        bulk_g2s(C + (size_t)p.plan.capr * row, ly.vc + off, (unsigned)nold * row, bar);
    }
}

// The kept experts' down rows of this CTA's output rows [o0, o1): expert slot j's rows at j * rd.
__device__ __noinline__ void fill_down(const PersistCall& p, const PersistLayer& ly, const int* kid, unsigned char* C,
                                       uint64_t* bar) {
    const PersistDims& d = p.dims;
    const int o0 = min((int)blockIdx.x * p.plan.rd, d.D), o1 = min(o0 + p.plan.rd, d.D);
    mbar_arrive_expect_tx(bar, (unsigned)(o1 - o0) * (unsigned)d.K * (unsigned)(d.F + d.F / 8));
    if (o1 <= o0) return;
    const int cap = p.plan.rd * d.K;  // rows the region holds
    for (int j = 0; j < d.K; ++j) {
        int e = kid[j];
        if (e < 0 || e >= d.E) e = 0;  // cannot happen: ranks are a permutation of [0, E)
        // rows o0.. of expert e are global rows e * D + o; in the region they sit at j * rd + (o - o0)
        fill_rows(C, o0 - j * p.plan.rd, cap, ly.wd_q, ly.wd_s, (int64_t)e * d.D, o0, o1, d.F, bar);
    }
}

// The producer warp's program (lane 0): every fill in the order the stages use them, each after the compute warps have
// released its region: per layer O, the chosen experts' down rows (as soon as the routing is known), the next layer's
// q/k/v and router rows, then its cache rows.  Per region that is W: q/k/v(0), O(0), q/k/v(1), O(1), ...; C: cache(0),
// down(0), cache(1), ...; R: router(0), router(1), ....  At the end it waits (bounded) for its last fill of each region, so no copy lands after the CTA ends.
__device__ void producer(const PersistCall& p, int len, unsigned char* sm, PsSmall& s) {
    const PersistLayout& L = p.plan.lay;
    const int nl = p.dims.L;
    unsigned iw = 0, ic = 0, ir = 0;  // fills issued per region
    if (!s.dead) {
        fill_qkv(p, p.layers[0], sm + L.w, &s.bw);
        ++iw;
        fill_router(p, p.layers[0], sm + L.r, &s.br);
        ++ir;
        fill_cache(p, p.layers[0], len, sm + L.c, &s.bc);
        ++ic;
    }
    for (int l = 0; l < nl && !*(volatile int*)&s.dead; ++l) {
        const bool more = l + 1 < nl;
        if (!producer_wait(&s.ev_w, 2u * l + 1u, p.err, s)) break;  // q/k/v of layer l done
        fill_o(p, p.layers[l], sm + L.w, &s.bw);
        ++iw;
        // the down rows first: the down-and-combine waits for them right after gate-up, while the next layer's
        // q/k/v and router rows are not needed before the next layer begins (issued before, they slowed the router
        // stage they ran beside)
        if (!producer_wait(&s.ev_route, l + 1u, p.err, s)) break;  // routing of layer l known (the cache rows used)
        fill_down(p, p.layers[l], s.kid, sm + L.c, &s.bc);
        ++ic;
        if (more) {
            if (!producer_wait(&s.ev_w, 2u * l + 2u, p.err, s)) break;  // O of layer l done
            fill_qkv(p, p.layers[l + 1], sm + L.w, &s.bw);
            ++iw;
            if (!producer_wait(&s.ev_r, l + 1u, p.err, s)) break;  // router of layer l done
            fill_router(p, p.layers[l + 1], sm + L.r, &s.br);
            ++ir;
            if (!producer_wait(&s.ev_c, l + 1u, p.err, s)) break;  // down-and-combine of layer l done
            fill_cache(p, p.layers[l + 1], len, sm + L.c, &s.bc);
            ++ic;
        }
    }
    if (iw) mbar_wait(&s.bw, (iw - 1) & 1, nullptr);
    if (ic) mbar_wait(&s.bc, (ic - 1) & 1, nullptr);
    if (ir) mbar_wait(&s.br, (ir - 1) & 1, nullptr);
}

// ---- shared pieces of the stages ------------------------------------------------------------------------------------

// The one-word quantizer of N independent blocks (warp-wide, block i's value of this lane in v[i]) with the same
// results as the projection kernels' (d = amax / 127, q = round-half-away(v / d), the IEEE quotient deciding near a
// half-integer); the rare IEEE division is out of line, which keeps the kernel's code short.
__device__ __noinline__ float ps_div_rn(float v, float d) { return __fdiv_rn(v, d); }

template <int N>
__device__ __forceinline__ void ps_quantize(const float (&v)[N], int8_t (&q)[N], float (&d)[N]) {
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
    if (__any_sync(0xffffffffu, near)) {
#pragma unroll 1
        for (int i = 0; i < N; ++i)
            if (quotient_near_tie(t[i], d[i])) t[i] = ps_div_rn(v[i], d[i]);
    }
#pragma unroll
    for (int i = 0; i < N; ++i)
        q[i] = d[i] == 0.0f ? (int8_t)0 : (int8_t)(int)fminf(fmaxf(roundf(t[i]), -127.0f), 127.0f);
}

// RMSNorm of the row a (written by other CTAs: read through L2) times w, quantized per 32-value block into the
// activation words (and low words) and scales in shared memory; every CTA forms the same values in the same order.
// Compute thread t holds values t + 352 j (a warp holds whole blocks); the squares are summed as f32 pairs and each y
// is rounded once.  With `copy`, CTA 0 also writes the row there (and to `copy2`).
template <int MODE, int NP>
__device__ __noinline__ void norm_quant(const float* a, const float* w, int D, float eps, int8_t* xq, int8_t* xl, float* xs,
                           PsSmall& s, float* copy, float* copy2) {
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    float av[NP], nw[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        const int i = t + PS_CT * j;
        nw[j] = i < D ? __ldg(w + i) : 0.f;
        av[j] = i < D ? __ldcg(a + i) : 0.f;
    }
    F2 ss = f2_two_prod(av[0], av[0]);
#pragma unroll
    for (int j = 1; j < NP; ++j) ss = f2_add(ss, f2_two_prod(av[j], av[j]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        ss = f2_add(ss, F2{__shfl_xor_sync(0xffffffffu, ss.hi, o), __shfl_xor_sync(0xffffffffu, ss.lo, o)});
    if (lane == 0) s.nred[wid] = ss;
    cbar();
    if (wid == 0) {  // the warps' sums in a fixed tree (lanes 0..14 hold them)
        F2 v = lane < PS_CW ? s.nred[lane] : F2{0.f, 0.f};
#pragma unroll
        for (int o = 8; o > 0; o >>= 1)
            v = f2_add(v, F2{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)});
        if (lane == 0) {
            const float df = (float)D;
            const float qh = v.hi / df;
            const float ql = (fmaf(-qh, df, v.hi) + v.lo) / df;
            s.nred[PS_CW] = f2_rsqrt(f2_add(f2_quick(qh, ql), F2{eps, 0.f}));
        }
    }
    cbar();
    const F2 inv = s.nred[PS_CW];
    float y[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        const int i = t + PS_CT * j;
        y[j] = f2_mul3_round(av[j], nw[j], inv);
        if (copy && blockIdx.x == 0 && i < D) {
            copy[i] = av[j];
            if (copy2) copy2[i] = av[j];
        }
    }
    int8_t qv[NP], lv[NP];
    float dsc[NP];
    if (MODE == 2) quantize2_lanes<NP>(y, qv, lv, dsc);  // round j: warp w holds block w + 11 j
    else ps_quantize<NP>(y, qv, dsc);
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        const int i = t + PS_CT * j;
        if (i < D) {
            xq[i] = qv[j];
            if (MODE == 2) xl[i] = lv[j];
            if (lane == 0) xs[i / 32] = dsc[j];
        }
    }
    cbar();
}

// A lane's activation blocks b = lane + 32 j (j < XB) in registers: words (and low words) and scales; zero past nb.
template <int MODE, int XB>
struct XRegs {
    uint32_t w[XB][8];
    uint32_t l[MODE == 2 ? XB : 1][8];
    float s[XB];
};

template <int MODE, int XB>
__device__ __forceinline__ void xregs_load(XRegs<MODE, XB>& x, const int8_t* xq, const int8_t* xl, const float* xs,
                                           int nb) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < XB; ++j) {
        const int b = lane + 32 * j;
        if (b < nb) {
            load_words32(xq + 32 * b, x.w[j]);
            if (MODE == 2) load_words32(xl + 32 * b, x.l[MODE == 2 ? j : 0]);
            x.s[j] = xs[b];
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

// A 32-byte block from shared memory, its two 16-byte halves read in an order that puts the eight lanes of a
// shared-memory phase (consecutive blocks, 32 bytes apart) on eight different 4-bank groups.
__device__ __forceinline__ void lds_block(const int8_t* p, uint32_t (&w)[8]) {
    const int sw = (threadIdx.x >> 2) & 1;
    const uint4* q = reinterpret_cast<const uint4*>(p);
    const uint4 a = q[sw], b = q[sw ^ 1];
    const uint4 lo = sw ? b : a, hi = sw ? a : b;
    w[0] = lo.x;
    w[1] = lo.y;
    w[2] = lo.z;
    w[3] = lo.w;
    w[4] = hi.x;
    w[5] = hi.y;
    w[6] = hi.z;
    w[7] = hi.w;
}

// R weight rows in shared memory (row r's quants at wq + r qstride, scales at ws + r sstride; rows past nvalid
// skipped) against the lane's activation blocks: lane takes blocks lane + 32 j in order, each block's exact int32 dot
// scaled by both scales (and 1/128 for the two-word dot) and added in f32; then each row's warp sum.
template <int MODE, int XB, int R>
__device__ __forceinline__ void row_dots(const int8_t* wq, int qstride, const float* ws, int sstride, int nb,
                                         int nvalid, const XRegs<MODE, XB>& x, float (&out)[R]) {
    const int lane = threadIdx.x & 31;
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.f;
#pragma unroll
    for (int j = 0; j < XB; ++j) {
        const int b = lane + 32 * j;
        if (b < nb) {
            uint32_t w[R][8];
            float sw[R];
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (r < nvalid) {
                    load_words32(wq + r * qstride + 32 * b, w[r]);
                    sw[r] = ws[r * sstride + b];
                }
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (r < nvalid) {
                    if (MODE == 2)
                        acc[r] = fmaf(sw[r] * x.s[j] * 0.0078125f,
                                      (float)block_dot_i8x2(w[r], x.w[j], x.l[MODE == 2 ? j : 0]), acc[r]);
                    else
                        acc[r] = fmaf(sw[r] * x.s[j], (float)block_dot_i8(w[r], x.w[j]), acc[r]);
                }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
#pragma unroll
    for (int r = 0; r < R; ++r) out[r] = acc[r];
}

// Ranking key: a NaN logit ranks below every number (and ties with -inf, broken by index).
__device__ __forceinline__ float ps_rank_key(float v) { return v != v ? -INFINITY : v; }

// The fold of one item (query head h, 32-dim quarter qd) of the attention partials: out = sum_j f_j o_j / sum_j f_j l_j
// with f_j = exp(m_j - max m).  Every warp holds the partials' maxima in its lanes (partial j in lane j % 32) and forms
// the max by shuffles; lane d of warp w sums f_j o_j[d] over the partials j = w, w + 11, ... in order, and the warps'
// sums meet in shared memory; warp 0 forms the denominator the same way.  The quarter is one 32-value block of the O
// projection's activation, quantized by warp 0.
template <int MODE>
__device__ void fold_item(const PersistCall& p, unsigned char* sm, PsSmall& s, int h, int qd) {
    constexpr int NU = (PS_MAXPPG + PS_CW - 1) / PS_CW;
    const PersistLayout& L = p.plan.lay;
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int ppg = p.plan.ppg;
    float* fr = smp<float>(sm, (uint32_t)(L.u + L.f_red));
    const float* base = p.part + (int64_t)h * ppg * (PS_HD + 2);
    float ov[NU];
#pragma unroll
    for (int u = 0; u < NU; ++u) {
        const int jj = wid + PS_CW * u;
        ov[u] = jj < ppg ? __ldcg(base + (int64_t)jj * (PS_HD + 2) + qd * 32 + lane) : 0.f;
    }
    const float m0 = lane < ppg ? __ldcg(base + (int64_t)lane * (PS_HD + 2) + PS_HD) : -FLT_MAX;
    const float m1 = lane + 32 < ppg ? __ldcg(base + (int64_t)(lane + 32) * (PS_HD + 2) + PS_HD) : -FLT_MAX;
    float l0 = 0.f, l1 = 0.f;
    if (wid == 0) {
        l0 = lane < ppg ? __ldcg(base + (int64_t)lane * (PS_HD + 2) + PS_HD + 1) : 0.f;
        l1 = lane + 32 < ppg ? __ldcg(base + (int64_t)(lane + 32) * (PS_HD + 2) + PS_HD + 1) : 0.f;
    }
    const float M = warp_max(fmaxf(m0, m1));
    float num = 0.f;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
        const int jj = wid + PS_CW * u;  // warp-uniform
        const float mj = __shfl_sync(0xffffffffu, jj < 32 ? m0 : m1, jj & 31);
        if (jj < ppg) num = fmaf(mj == -FLT_MAX ? 0.f : expf(mj - M), ov[u], num);
    }
    fr[wid * 32 + lane] = num;
    if (wid == 0) {
        float den = (m0 == -FLT_MAX ? 0.f : expf(m0 - M)) * l0;
        den = fmaf(m1 == -FLT_MAX ? 0.f : expf(m1 - M), l1, den);
        den = group_sum<32>(den);
        if (lane == 0) s.den = den;
    }
    cbar();
    if (wid == 0) {
        float o = 0.f;
#pragma unroll
        for (int v = 0; v < PS_CW; ++v) o += fr[v * 32 + lane];
        const float den = s.den;
        o = den > 0.f ? o / den : 0.f;
        const int64_t oi = (int64_t)h * PS_HD + qd * 32 + lane;
        p.att[oi] = o;
        float dsc;
        if (MODE == 2) {
            int8_t lv;
            p.attq[oi] = quantize2_lane(o, dsc, lv);
            p.attl[oi] = lv;
        } else {
            const float ov1[1] = {o};
            int8_t q1[1];
            float d1[1];
            ps_quantize<1>(ov1, q1, d1);
            p.attq[oi] = q1[0];
            dsc = d1[0];
        }
        if (lane == 0) p.atts[oi / 32] = dsc;
    }
    cbar();
}

// The fold of a key/value head's partials inside the attention stage, by the last CTAs of the head to finish: each CTA
// of head g takes a ticket when its partials are written (an arrival counter per head that only grows within a launch);
// ticket t of the layer folds the items i = ppg - 1 - t, + ppg, ... (the last arriver item 0), once every CTA of the head
// has arrived (a bounded wait).  Items: (query head of the group, 32-dim quarter).
template <int MODE>
__device__ void fold_tail(const PersistCall& p, unsigned char* sm, PsSmall& s, int l, int g) {
    const PersistDims& d = p.dims;
    const int G = d.H / d.KV, ppg = p.plan.ppg, nit = G * 4;
    unsigned* cnt = p.bar + PS_GROUP_BAR + g * PS_BAR_STRIDE;
    cbar();  // this CTA's partials are written
    if (threadIdx.x == 0) s.ticket = (int)(atom_add_acq_rel_u32(cnt, 1u) - (unsigned)l * ppg);
    cbar();
    const int first = ppg - 1 - s.ticket;
    if (first < 0 || first >= nit) return;  // CTA-uniform
    if (threadIdx.x == 0 && !s.dead) {
        const unsigned target = (unsigned)(l + 1) * ppg;
        const long long t0 = clock64();
        while ((int)(ld_acquire_gpu(cnt) - target) < 0) {
            if (clock64() - t0 > kGridWaitCycles || (*(volatile int*)p.err & kErrPipeline)) {
                atomicOr(p.err, kErrPipeline);
                s.dead = 1;
                break;
            }
        }
    }
    cbar();
    for (int i = first; i < nit; i += ppg) fold_item<MODE>(p, sm, s, g * G + i / 4, i % 4);
}

// ---- the stages (compute warps) -------------------------------------------------------------------------------------

// A: the attention norm (layer 0: of the token's embedding row, which becomes the residual) and this CTA's q/k/v rows:
// warp w takes rows w, w + 11, w + 22, ... three at a time, the activation blocks in registers.
template <int MODE, int BPL, int NP>
__device__ void stage_qkv(const PersistCall& p, const PersistLayer& ly, int l, unsigned char* sm, PsSmall& s,
                          unsigned& nw) {
    const PersistDims& d = p.dims;
    const PersistLayout& L = p.plan.lay;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int8_t* xq = smp<int8_t>(sm, (uint32_t)(L.xq));
    int8_t* xl = smp<int8_t>(sm, (uint32_t)(L.xl));
    float* xs = smp<float>(sm, (uint32_t)(L.xs));
    const float* a = p.h;
    if (l == 0) {
        const int32_t tok = *p.tok;
        const bool bad = tok < 0 || tok >= p.vocab;  // an out-of-range token: flagged, row 0 read instead
        if (bad && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.err, 1);
        a = p.embed + (int64_t)(bad ? 0 : tok) * d.D;
    }
    norm_quant<MODE, NP>(a, ly.attn_norm, d.D, p.eps, xq, xl, xs, s, l == 0 ? p.h : nullptr,
                         l == 0 ? p.trace : nullptr);
    const int nb = d.D / 32;
    XRegs<MODE, BPL> x;
    xregs_load<MODE, BPL>(x, xq, xl, xs, nb);
    region_wait(&s.bw, nw, p.err, s);
    const int NQ = d.H * PS_HD, NK = d.KV * PS_HD, NR = NQ + 2 * NK;
    const int r0 = min((int)blockIdx.x * p.plan.rq, NR), r1 = min(r0 + p.plan.rq, NR);
    const int8_t* W = smp<const int8_t>(sm, (uint32_t)(L.w));
    const float* Ws = smp<const float>(sm, (uint32_t)(L.w + (size_t)p.plan.rq * d.D));
    for (int i = wid; i < r1 - r0; i += 3 * PS_CW) {
        float v[3];
        const int nv = min(3, (r1 - r0 - i + PS_CW - 1) / PS_CW);
        row_dots<MODE, BPL, 3>(W + (size_t)i * d.D, PS_CW * d.D, Ws + (size_t)i * nb, PS_CW * nb, nb, nv, x, v);
        if (lane == 0)
#pragma unroll
            for (int u = 0; u < 3; ++u)
                if (u < nv) {
                    const int r = r0 + i + u * PS_CW;
                    float* dst = r < NQ ? p.q + r : r < NQ + NK ? p.k + (r - NQ) : p.v + (r - NQ - NK);
                    *dst = v[u];
                }
    }
}

// P: this CTA's positions of its key/value head for every query head of the group.
//   QK-norm + RoPE: warp h < G turns query head h, warp G the new key and warp G + 1 takes the new value (the CTA that
//   holds the new position); lane l the pairs (l, l + 64) and (l + 32, l + 96).
//   Scores: warp w takes positions w, w + 11, ...; lane (head pair l >> 3, dim group l & 7) holds its two heads' dims
//   4 (l & 7) + 32 i .. + 3 (i < 4) in registers, so a key row is read once per warp, each 16-byte piece by the four
//   lanes of a group at once; the dim groups' sums meet by shuffles.
//   Values: warp w takes the same positions, lane l the dims 4 l .. 4 l + 3 of every head (32 sums in registers); the
//   11 warps' sums meet in shared memory in a fixed order (warp w + 8 into warp w, then warps 0..7 in order).
template <int MODE>
__device__ void stage_attention(const PersistCall& p, const PersistLayer& ly, int l, int len, unsigned char* sm,
                                PsSmall& s, unsigned& nc) {
    const PersistDims& d = p.dims;
    const PersistLayout& L = p.plan.lay;
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int G = d.H / d.KV, capr = p.plan.capr;
    int g, p0, np;
    attn_share(p, len, g, p0, np);
    const int pos = len - 1;
    const bool has_new = np > 0 && p0 + np == len;  // CTA-uniform
    float* qs = smp<float>(sm, (uint32_t)(L.u + L.b_qs));
    float* kn = smp<float>(sm, (uint32_t)(L.u + L.b_kn));
    float* vn = smp<float>(sm, (uint32_t)(L.u + L.b_vn));
    float* sc = smp<float>(sm, (uint32_t)(L.u + L.b_sc));  // [position][PS_MAXG]
    float* red = smp<float>(sm, (uint32_t)((L.red_in_c ? L.c : L.u) + L.b_red));
    if (np > 0 && wid < G + 2) {
        const float* src = nullptr;
        const float* nw = nullptr;
        if (wid < G) {
            src = p.q + ((int64_t)g * G + wid) * PS_HD;
            nw = ly.q_norm;
        } else if (has_new) {
            src = (wid == G ? p.k : p.v) + (int64_t)g * PS_HD;
            nw = wid == G ? ly.k_norm : nullptr;
        }
        if (src) {
            const float a0 = __ldcg(src + lane), b0 = __ldcg(src + lane + 64);
            const float a1 = __ldcg(src + lane + 32), b1 = __ldcg(src + lane + 96);
            float o0, o1, o2, o3;  // dims lane, lane + 64, lane + 32, lane + 96
            if (nw) {  // RMSNorm (eps inside the root, the head weight multiplies), then the NeoX rotation of (i, i + 64)
                const float ss = group_sum<32>((a0 * a0 + b0 * b0) + (a1 * a1 + b1 * b1));
                const float inv = 1.0f / sqrtf(ss / (float)PS_HD + p.eps);
                const float* ct = p.cos_t + (int64_t)pos * (PS_HD / 2);
                const float* st = p.sin_t + (int64_t)pos * (PS_HD / 2);
                const float c0 = __ldg(ct + lane), s0 = __ldg(st + lane), c1 = __ldg(ct + lane + 32), s1 = __ldg(st + lane + 32);
                const float x0 = a0 * inv * __ldg(nw + lane), y0 = b0 * inv * __ldg(nw + lane + 64);
                const float x1 = a1 * inv * __ldg(nw + lane + 32), y1 = b1 * inv * __ldg(nw + lane + 96);
                o0 = x0 * c0 - y0 * s0;
                o1 = x0 * s0 + y0 * c0;
                o2 = x1 * c1 - y1 * s1;
                o3 = x1 * s1 + y1 * c1;
            } else {
                o0 = a0;
                o1 = b0;
                o2 = a1;
                o3 = b1;
            }
            float* dst = wid < G ? qs + wid * PS_HD : wid == G ? kn : vn;
            dst[lane] = o0;
            dst[lane + 64] = o1;
            dst[lane + 32] = o2;
            dst[lane + 96] = o3;
            if (wid >= G) {  // the new key or value row into the cache
                float* out = (wid == G ? ly.kc : ly.vc) + ((int64_t)g * d.ctx + pos) * PS_HD;
                out[lane] = o0;
                out[lane + 64] = o1;
                out[lane + 32] = o2;
                out[lane + 96] = o3;
            }
        }
    }
    region_wait(&s.bc, nc, p.err, s);  // the staged cache rows (its CTA barrier also publishes the rows above)
    if (np > 0) {
        const float* Kc = smp<const float>(sm, (uint32_t)(L.c));
        const float* Vc = Kc + (size_t)capr * PS_HD;
        {
            const int hp = lane >> 3, gq = lane & 7;
            const int h0 = 2 * hp, h1 = 2 * hp + 1;
            float q0[16], q1[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 a = h0 < G ? *reinterpret_cast<const float4*>(qs + h0 * PS_HD + 32 * i + 4 * gq)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 b = h1 < G ? *reinterpret_cast<const float4*>(qs + h1 * PS_HD + 32 * i + 4 * gq)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                q0[4 * i] = a.x;
                q0[4 * i + 1] = a.y;
                q0[4 * i + 2] = a.z;
                q0[4 * i + 3] = a.w;
                q1[4 * i] = b.x;
                q1[4 * i + 1] = b.y;
                q1[4 * i + 2] = b.z;
                q1[4 * i + 3] = b.w;
            }
#pragma unroll 2
            for (int pl = wid; pl < np; pl += PS_CW) {
                const float* krow = (has_new && pl == np - 1) ? kn : Kc + (size_t)pl * PS_HD;
                float s0a = 0.f, s0b = 0.f, s1a = 0.f, s1b = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 k4 = *reinterpret_cast<const float4*>(krow + 32 * i + 4 * gq);
                    float& s0 = i < 2 ? s0a : s0b;
                    float& s1 = i < 2 ? s1a : s1b;
                    s0 = fmaf(q0[4 * i], k4.x, s0);
                    s0 = fmaf(q0[4 * i + 1], k4.y, s0);
                    s0 = fmaf(q0[4 * i + 2], k4.z, s0);
                    s0 = fmaf(q0[4 * i + 3], k4.w, s0);
                    s1 = fmaf(q1[4 * i], k4.x, s1);
                    s1 = fmaf(q1[4 * i + 1], k4.y, s1);
                    s1 = fmaf(q1[4 * i + 2], k4.z, s1);
                    s1 = fmaf(q1[4 * i + 3], k4.w, s1);
                }
                float s0 = s0a + s0b, s1 = s1a + s1b;
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    s0 += __shfl_xor_sync(0xffffffffu, s0, o);
                    s1 += __shfl_xor_sync(0xffffffffu, s1, o);
                }
                if (gq == 0) {
                    if (h0 < G) sc[pl * PS_MAXG + h0] = s0 * p.scale;
                    if (h1 < G) sc[pl * PS_MAXG + h1] = s1 * p.scale;
                }
            }
        }
        cbar();
        // the share's softmax statistics per head (warp hh), scores replaced by exp(s - m)
        for (int hh = wid; hh < G; hh += PS_CW) {
            float m = -FLT_MAX;
            for (int i = lane; i < np; i += 32) m = fmaxf(m, sc[i * PS_MAXG + hh]);
            m = warp_max(m);
            float lsum = 0.f;
            for (int i = lane; i < np; i += 32) {
                const float e = expf(sc[i * PS_MAXG + hh] - m);
                sc[i * PS_MAXG + hh] = e;
                lsum += e;
            }
            lsum = group_sum<32>(lsum);
            if (lane == 0) {
                s.stat[hh][0] = m;
                s.stat[hh][1] = lsum;
            }
        }
        cbar();
        float4 acc[PS_MAXG];
#pragma unroll
        for (int h = 0; h < PS_MAXG; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
        for (int pl = wid; pl < np; pl += PS_CW) {
            const float4 v4 = (has_new && pl == np - 1) ? reinterpret_cast<const float4*>(vn)[lane]
                                                        : reinterpret_cast<const float4*>(Vc + (size_t)pl * PS_HD)[lane];
            const float4 e0 = *reinterpret_cast<const float4*>(sc + pl * PS_MAXG);
            const float4 e1 = *reinterpret_cast<const float4*>(sc + pl * PS_MAXG + 4);
            const float e[PS_MAXG] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
            for (int h = 0; h < PS_MAXG; ++h)
                if (h < G) {
                    acc[h].x = fmaf(e[h], v4.x, acc[h].x);
                    acc[h].y = fmaf(e[h], v4.y, acc[h].y);
                    acc[h].z = fmaf(e[h], v4.z, acc[h].z);
                    acc[h].w = fmaf(e[h], v4.w, acc[h].w);
                }
        }
        float4* r4 = reinterpret_cast<float4*>(red);  // [PS_PVW][G][32 lanes]
        if (wid >= PS_PVW)
#pragma unroll
            for (int h = 0; h < PS_MAXG; ++h)
                if (h < G) r4[((wid - PS_PVW) * G + h) * 32 + lane] = acc[h];
        cbar();
        if (wid < PS_CW - PS_PVW)
#pragma unroll
            for (int h = 0; h < PS_MAXG; ++h)
                if (h < G) {
                    const float4 o = r4[(wid * G + h) * 32 + lane];
                    acc[h].x += o.x;
                    acc[h].y += o.y;
                    acc[h].z += o.z;
                    acc[h].w += o.w;
                }
        cbar();
        if (wid < PS_PVW)
#pragma unroll
            for (int h = 0; h < PS_MAXG; ++h)
                if (h < G) r4[(wid * G + h) * 32 + lane] = acc[h];
        cbar();
    }
    if (g < d.KV) {  // the partial (an empty share weighs nothing: max -FLT_MAX, sum 0)
        const int j = (int)blockIdx.x % p.plan.ppg;
        for (int i = t; i < G * PS_HD; i += PS_CT) {
            const int hh = i / PS_HD, dd = i % PS_HD;
            float o = 0.f;
            if (np > 0) {
                o = red[hh * PS_HD + dd];
#pragma unroll
                for (int w = 1; w < PS_PVW; ++w) o += red[(w * G + hh) * PS_HD + dd];
            }
            p.part[(((int64_t)g * G + hh) * p.plan.ppg + j) * (PS_HD + 2) + dd] = o;
        }
        if (t < G) {
            float* b = p.part + (((int64_t)g * G + t) * p.plan.ppg + j) * (PS_HD + 2);
            b[PS_HD] = np > 0 ? s.stat[t][0] : -FLT_MAX;
            b[PS_HD + 1] = np > 0 ? s.stat[t][1] : 0.f;
        }
        fold_tail<MODE>(p, sm, s, l, g);
    }
}

// O: the attention output's words staged in shared memory, then this CTA's O rows (warp w: row w, w + 11, ...) with
// the residual add (in place: every CTA read the residual row before the first barrier of the layer).
template <int MODE>
__device__ void stage_o(const PersistCall& p, unsigned char* sm, PsSmall& s, unsigned& nw) {
    constexpr int XB = PS_MAXHHD / 1024;
    const PersistDims& d = p.dims;
    const PersistLayout& L = p.plan.lay;
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int HHD = d.H * PS_HD, nbo = HHD / 32;
    int8_t* oq = smp<int8_t>(sm, (uint32_t)(L.u + L.o_q));
    int8_t* ol = smp<int8_t>(sm, (uint32_t)(L.u + L.o_l));
    float* os = smp<float>(sm, (uint32_t)(L.u + L.o_s));
    for (int i = t; i < HHD / 16; i += PS_CT) {
        reinterpret_cast<uint4*>(oq)[i] = __ldcg(reinterpret_cast<const uint4*>(p.attq) + i);
        if (MODE == 2) reinterpret_cast<uint4*>(ol)[i] = __ldcg(reinterpret_cast<const uint4*>(p.attl) + i);
    }
    for (int i = t; i < nbo; i += PS_CT) os[i] = __ldcg(p.atts + i);
    region_wait(&s.bw, nw, p.err, s);  // (its CTA barrier also publishes the staged words)
    XRegs<MODE, XB> x;
    xregs_load<MODE, XB>(x, oq, ol, os, nbo);
    const int r0 = min((int)blockIdx.x * p.plan.ro, d.D), r1 = min(r0 + p.plan.ro, d.D);
    const int8_t* W = smp<const int8_t>(sm, (uint32_t)(L.w));
    const float* Ws = smp<const float>(sm, (uint32_t)(L.w + (size_t)p.plan.ro * HHD));
    for (int i = wid; i < r1 - r0; i += PS_CW) {
        float v[1];
        row_dots<MODE, XB, 1>(W + (size_t)i * HHD, 0, Ws + (size_t)i * nbo, 0, nbo, 1, x, v);
        if (lane == 0) {
            const int o = r0 + i;
            p.h[o] = __ldcg(p.h + o) + v[0];
        }
    }
}

// R: the mixture's norm (the words stay in shared memory for gate-up) and this CTA's router rows.
template <int MODE, int BPL, int NP>
__device__ void stage_router(const PersistCall& p, const PersistLayer& ly, unsigned char* sm, PsSmall& s, unsigned& nr) {
    const PersistDims& d = p.dims;
    const PersistLayout& L = p.plan.lay;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int8_t* xq = smp<int8_t>(sm, (uint32_t)(L.xq));
    int8_t* xl = smp<int8_t>(sm, (uint32_t)(L.xl));
    float* xs = smp<float>(sm, (uint32_t)(L.xs));
    norm_quant<MODE, NP>(p.h, ly.ffn_norm, d.D, p.eps, xq, xl, xs, s, nullptr, nullptr);
    const int e0 = min((int)blockIdx.x * p.plan.rr, d.E), e1 = min(e0 + p.plan.rr, d.E);
    const int nb = d.D / 32;
    XRegs<MODE, BPL> x;
    if (wid < e1 - e0) xregs_load<MODE, BPL>(x, xq, xl, xs, nb);
    region_wait(&s.br, nr, p.err, s);
    const int8_t* R = smp<const int8_t>(sm, (uint32_t)(L.r));
    const float* Rs = smp<const float>(sm, (uint32_t)(L.r + (size_t)p.plan.rr * d.D));
    for (int i = wid; i < e1 - e0; i += PS_CW) {
        float v[1];
        row_dots<MODE, BPL, 1>(R + (size_t)i * d.D, 0, Rs + (size_t)i * nb, 0, nb, 1, x, v);
        if (lane == 0) p.logits[e0 + i] = v[0];
    }
}

// E: every CTA ranks the logits (expert e's place = the experts with a larger key, or an equal key and a lower index)
// and forms the gates (softmax over all experts renormalized over the kept = softmax over the kept logits), which lets
// the producer request the chosen experts' down rows; then this CTA's gate-up items (kept expert j, hidden row i)
// stream into registers: warp w takes a consecutive range of items, IPW at a time with all their loads in flight before any is
// used, then arrives on the 32-row blocks of its range (the warp completing a block quantizes it).
template <int MODE, int BPL>
__device__ void stage_gate_up(const PersistCall& p, const PersistLayer& ly, int l, unsigned char* sm, PsSmall& s) {
    constexpr int IPW = BPL >= 4 ? 1 : 2;
    const PersistDims& d = p.dims;
    const PersistLayout& L = p.plan.lay;
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    float* key = smp<float>(sm, (uint32_t)(L.u + L.e_key));
    float* val = smp<float>(sm, (uint32_t)(L.u + L.e_val));
    const int E8 = (d.E + 7) & ~7;
    for (int e = t; e < E8; e += PS_CT) {
        const float v = e < d.E ? __ldcg(p.logits + e) : 0.f;
        val[e] = v;
        key[e] = e < d.E ? ps_rank_key(v) : -INFINITY;  // padding never counts: it sits past every real index
    }
    cbar();
    for (int e = t; e < d.E; e += PS_CT) {
        const float ke = key[e];
        int r = 0;
        for (int f = 0; f < E8; f += 4) {
            const float4 a = *reinterpret_cast<const float4*>(key + f);
            r += (a.x > ke) || (a.x == ke && f < e);
            r += (a.y > ke) || (a.y == ke && f + 1 < e);
            r += (a.z > ke) || (a.z == ke && f + 2 < e);
            r += (a.w > ke) || (a.w == ke && f + 3 < e);
        }
        if (r < d.K) {
            s.kid[r] = e;
            s.kval[r] = val[e];
        }
    }
    cbar();
    signal(&s.ev_route, (unsigned)l + 1u);  // the kept experts are known: their down rows may come
    if (wid == 0) {
        const float kept = lane < d.K ? s.kval[lane] : 0.f;
        const float m = s.kval[0];
        const float pe = lane < d.K ? expf(kept - m) : 0.f;
        const float z = group_sum<32>(pe);
        if (lane < d.K) {
            const float gt = __fdiv_rn(pe, z);
            s.gate[lane] = gt;
            if (blockIdx.x == 0) {
                p.ids[lane] = s.kid[lane];
                p.gates[lane] = gt;
            }
        }
    }
    int bidx[BPL];
    bool bval[BPL];
    const int nb = d.D / 32;
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        bidx[j] = lane + 32 * j;
        bval[j] = bidx[j] < nb;
    }
    XTile<MODE, BPL> x;
    load_x<MODE, BPL>(x, nullptr, smp<const int8_t>(sm, (uint32_t)(L.xq)), smp<const int8_t>(sm, (uint32_t)(L.xl)),
                      smp<const float>(sm, (uint32_t)(L.xs)), bidx, bval);
    const int nk = d.K * d.F;
    const int i0 = min((int)blockIdx.x * p.plan.gu, nk), i1 = min(i0 + p.plan.gu, nk);
    // warp w's items are the consecutive range [w0, w1), IPW at a time
    const int per = (i1 - i0 + PS_CW - 1) / PS_CW;
    const int w0 = min(i0 + wid * per, i1), w1 = min(w0 + per, i1);
    for (int it0 = w0; it0 < w1; it0 += IPW) {
        WTile<BPL, 1> tg[IPW], tu[IPW];
#pragma unroll
        for (int u = 0; u < IPW; ++u) {
            const int it = it0 + u;
            const bool v = it < w1;
            const int jx = v ? it / d.F : 0;
            const int i = v ? it - jx * d.F : 0;
            const int64_t row = (int64_t)s.kid[jx] * d.F + i;
            load_tile<BPL, 1>(tg[u], ly.wg_q, ly.wg_s, row, v ? 1 : 0, d.D, nb, bidx, bval);
            load_tile<BPL, 1>(tu[u], ly.wu_q, ly.wu_s, row, v ? 1 : 0, d.D, nb, bidx, bval);
        }
#pragma unroll
        for (int u = 0; u < IPW; ++u) {
            const float gv = group_sum<32>(tile_row_dot<MODE, BPL, 1>(tg[u], 0, x));
            const float uv = group_sum<32>(tile_row_dot<MODE, BPL, 1>(tu[u], 0, x));
            if (lane == 0 && it0 + u < w1) p.hbuf[it0 + u] = silu_f32(gv) * uv;
        }
    }
    // the int8 epilogue: the warp arrives on the 32-row blocks its items belong to, releasing its rows; the warp that
    // completes a block quantizes it (lane = row) and leaves the block's counter at zero
    for (int b = w0 / 32; w1 > w0 && b <= (w1 - 1) / 32; ++b) {
        const int lo = max(w0, b * 32), hi = min(w1 - 1, b * 32 + 31);
        int old = 0;
        __syncwarp();
        if (lane == 0) old = atomic_add_acq_rel_gpu(p.qcnt + b, hi - lo + 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old + (hi - lo + 1) == 32) {  // warp-uniform
            __syncwarp();
            const float hv = __ldcg(p.hbuf + (int64_t)b * 32 + lane);
            float dsc;
            if (MODE == 2) {
                int8_t lv;
                p.hq[(int64_t)b * 32 + lane] = quantize2_lane(hv, dsc, lv);
                p.hl[(int64_t)b * 32 + lane] = lv;
            } else {
                const float v1[1] = {hv};
                int8_t q1[1];
                float d1[1];
                ps_quantize<1>(v1, q1, d1);
                p.hq[(int64_t)b * 32 + lane] = q1[0];
                dsc = d1[0];
            }
            if (lane == 0) {
                p.hs[b] = dsc;
                p.qcnt[b] = 0;
            }
        }
    }
}

// D: every CTA stages the K hidden rows' words and scales (gate-up quantized each 32-row block); then its output rows o
// (warp w: rows w, w + 11, ...): y[o] = residual[o] + sum_j g_j (W_down[e_j] row o . h_j), the (expert, block) pairs
// dealt to the lanes in order, g_j (s_w s_x D) added in f32 per lane, then across the warp.  The rows come from the
// C region (the producer copied them there once the routing was known).
template <int MODE>
__device__ void stage_down(const PersistCall& p, int l, unsigned char* sm, PsSmall& s, unsigned& nc) {
    const PersistDims& d = p.dims;
    const PersistLayout& L = p.plan.lay;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int KF = d.K * d.F, NBH = KF / 32, nbf = d.F / 32;
    int8_t* hq = smp<int8_t>(sm, (uint32_t)(L.u + L.d_q));
    int8_t* hl = smp<int8_t>(sm, (uint32_t)(L.u + L.d_l));
    float* hs = smp<float>(sm, (uint32_t)(L.u + L.d_s));
    for (int i = threadIdx.x; i < KF / 16; i += PS_CT) {
        reinterpret_cast<uint4*>(hq)[i] = __ldcg(reinterpret_cast<const uint4*>(p.hq) + i);
        if (MODE == 2) reinterpret_cast<uint4*>(hl)[i] = __ldcg(reinterpret_cast<const uint4*>(p.hl) + i);
    }
    for (int i = threadIdx.x; i < NBH; i += PS_CT) hs[i] = __ldcg(p.hs + i);
    region_wait(&s.bc, nc, p.err, s);  // (its CTA barrier also publishes the words)
    const int o0 = min((int)blockIdx.x * p.plan.rd, d.D), o1 = min(o0 + p.plan.rd, d.D);
    const int8_t* C = smp<const int8_t>(sm, (uint32_t)(L.c));
    const float* Cs = smp<const float>(sm, (uint32_t)(L.c + (size_t)p.plan.rd * d.K * d.F));
    const int P = d.K * nbf;
    for (int i = wid; i < o1 - o0; i += PS_CW) {
        const float res = __ldcg(p.h + o0 + i);
        float acc = 0.f;
        int jx = lane / nbf, b = lane - jx * nbf;  // pair pi = jx nbf + b, advanced 32 pairs at a time
        for (int pb = lane; pb < P; pb += 32) {
            const int rr = jx * p.plan.rd + i;  // the row's place in the staged rows
            uint32_t w[8], x[8];
            lds_block(C + rr * d.F + 32 * b, w);
            lds_block(hq + jx * d.F + 32 * b, x);
            if (MODE == 2) {
                uint32_t x2[8];
                lds_block(hl + jx * d.F + 32 * b, x2);
                acc = fmaf(s.gate[jx] * (Cs[rr * nbf + b] * hs[jx * nbf + b] * 0.0078125f),
                           (float)block_dot_i8x2(w, x, x2), acc);
            } else {
                acc = fmaf(s.gate[jx] * (Cs[rr * nbf + b] * hs[jx * nbf + b]), (float)block_dot_i8(w, x), acc);
            }
            b += 32;
            while (b >= nbf) {
                b -= nbf;
                ++jx;
            }
        }
        acc = group_sum<32>(acc);
        if (lane == 0) {
            const int o = o0 + i;
            const float y = res + acc;
            p.h[o] = y;
            if (p.trace) p.trace[(int64_t)(l + 1) * d.D + o] = y;
        }
    }
}

// ---- the kernel -------------------------------------------------------------------------------------------------------

// grid = one CTA per SM (cooperative launch), 384 threads: warps 0..10 compute, warp 11 the producer.  BPL = 32-value
// blocks of a d-wide row per lane (d <= 1024 BPL); NP = 352-value rounds of the residual row per compute thread.
template <int MODE, int BPL>
__global__ void __maxnreg__(168) decode_persistent_kernel(const __grid_constant__ PersistCall p) {
    extern __shared__ __align__(128) unsigned char sm[];
    constexpr int NP = (1024 * BPL + PS_CT - 1) / PS_CT;
    PsSmall& s = *reinterpret_cast<PsSmall*>(sm);
    const int t = threadIdx.x;
    const int len = *p.pos + 1;  // the cache length this step, fixed for the launch
    if (t == 0) {
        mbar_init(&s.bw, 1);
        mbar_init(&s.bc, 1);
        mbar_init(&s.br, 1);
        s.ev_w = s.ev_r = s.ev_route = s.ev_c = 0;
        // after a wait gave up (an earlier launch's record is still in the error word) nothing waits at all
        s.dead = (*(volatile int*)p.err & kErrPipeline) ? 1 : 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (t >= PS_CT) {  // the producer warp: one lane issues every fill
        if (t == PS_CT) producer(p, len, sm, s);
        return;
    }
    if ((len < 1 || len > p.dims.ctx) && blockIdx.x == 0 && t == 0) atomicOr(p.err, 2);
    unsigned nw = 0, nc = 0, nr = 0;  // completed fills of each region (uniform over the compute warps)
    unsigned kb = 0;                  // grid barriers of this launch
#pragma unroll 1
    for (int li = 0; li < p.dims.L; ++li) {
        // an opaque copy of the layer index: the compiler keeps one body for every layer instead of peeling the first
        // and last (three copies of a large body do not fit the instruction cache)
        int l;
        asm volatile("mov.u32 %0, %1;" : "=r"(l) : "r"(li));
        const PersistLayer& ly = p.layers[l];
        const bool more = l + 1 < p.dims.L;
        // a region's next fill is released after the grid barrier that follows its last use: copies started just
        // before a barrier slow the barrier (the release and the arrivals queue behind them)
        stage_qkv<MODE, BPL, NP>(p, ly, l, sm, s, nw);
        grid_barrier(p.bar, kb++, p.err, s);
        signal(&s.ev_w, 2u * l + 1u);  // the W region's q/k/v rows are used: O may come
        stage_attention<MODE>(p, ly, l, len, sm, s, nc);
        grid_barrier(p.bar, kb++, p.err, s);
        stage_o<MODE>(p, sm, s, nw);
        grid_barrier(p.bar, kb++, p.err, s);
        signal(&s.ev_w, 2u * l + 2u);  // O's rows are used: the next layer's q/k/v may come
        stage_router<MODE, BPL, NP>(p, ly, sm, s, nr);
        grid_barrier(p.bar, kb++, p.err, s);
        signal(&s.ev_r, l + 1u);
        stage_gate_up<MODE, BPL>(p, ly, l, sm, s);
        grid_barrier(p.bar, kb++, p.err, s);
        stage_down<MODE>(p, l, sm, s, nc);
        if (more) {
            grid_barrier(p.bar, kb++, p.err, s);
            signal(&s.ev_c, l + 1u);  // the down rows are used: the next layer's cache rows may come
        }
    }
    cbar();
    // the last CTA out leaves the barrier counters at zero for the next launch
    if (t == 0 && !s.dead) {
        unsigned* exits = p.bar + PS_BARS * PS_BAR_STRIDE;
        const unsigned old = atom_add_acq_rel_u32(exits, 1u);
        if (old == gridDim.x - 1) {
            for (int i = 0; i < PS_BARS; ++i) atomicExch(p.bar + i * PS_BAR_STRIDE, 0u);
            for (int g = 0; g < p.dims.KV; ++g) atomicExch(p.bar + PS_GROUP_BAR + g * PS_BAR_STRIDE, 0u);
            atomicExch(exits, 0u);
        }
    }
}

template <int MODE, int BPL>
cudaError_t run_persist(const PersistCall& c, cudaStream_t st) {
    auto kern = decode_persistent_kernel<MODE, BPL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.plan.smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, PS_THREADS, c.plan.smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c.plan.nb);
    cfg.blockDim = dim3(PS_THREADS);
    cfg.dynamicSmemBytes = c.plan.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, c);
}

// Whether one CTA of the instance for these shapes fits an SM with `smem` bytes of shared memory.
template <int MODE, int BPL>
bool fits(size_t smem) {
    auto kern = decode_persistent_kernel<MODE, BPL>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return false;
    int occ = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, PS_THREADS, smem) == cudaSuccess && occ >= 1;
}

bool persist_fits(const PersistDims& d, size_t smem) {
    if (d.mode == 2) return d.D <= 1024 ? fits<2, 1>(smem) : d.D <= 2048 ? fits<2, 2>(smem) : fits<2, 4>(smem);
    return d.D <= 1024 ? fits<1, 1>(smem) : d.D <= 2048 ? fits<1, 2>(smem) : fits<1, 4>(smem);
}

}  // namespace

PersistPlan persist_plan(const PersistDims& d) {
    PersistPlan pl;
    auto no = [&](const char* why) {
        pl.ok = 0;
        pl.why = why;
        return pl;
    };
    if (d.mode != 1 && d.mode != 2) return no("the f32-activation mode");
    if (d.L < 1 || d.D < 128 || d.D % 128 || d.D > 4096) return no("d is not a multiple of 128 up to 4096");
    if (d.KV < 1 || d.H < 1 || d.H % d.KV || d.H / d.KV > PS_MAXG) return no("more than 8 query heads a key/value head");
    if (d.H * PS_HD > PS_MAXHHD) return no("more than 32 query heads");
    if (d.KV > PS_MAXKV) return no("more than 12 key/value heads");
    if (d.F < 128 || d.F % 128) return no("dff is not a multiple of 128");
    if (d.K < 1 || d.K > PS_MAXK || d.K > d.E || d.E > PS_MAXE) return no("top-k or expert count out of range");
    if (d.ctx < 1) return no("no cache");
    int dev = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
        return no("no cooperative launch on this device");
    const DeviceInfo& di = device_info();
    pl.nb = di.sms;
    pl.ppg = pl.nb / d.KV;
    if (pl.ppg < 1 || pl.ppg > PS_MAXPPG) return no("key/value heads do not match the SM count");
    auto cdiv = [](int64_t a, int64_t b) { return (int)((a + b - 1) / b); };
    pl.rq = cdiv((int64_t)(d.H + 2 * d.KV) * PS_HD, pl.nb);
    pl.ro = cdiv(d.D, pl.nb);
    pl.rr = cdiv(d.E, pl.nb);
    pl.rd = cdiv(d.D, pl.nb);
    pl.capr = cdiv(d.ctx, pl.ppg);
    pl.gu = cdiv((int64_t)d.K * d.F, pl.nb);
    pl.lay = ps_layout(d, pl);
    pl.smem = pl.lay.total;
    if ((int64_t)pl.smem > di.smem_optin) return no("the stages' shared memory does not fit (cache or rows per CTA)");
    if (!persist_fits(d, pl.smem)) return no("a CTA of the kernel does not fit an SM");
    pl.ok = 1;
    return pl;
}

cudaError_t launch_persist(const PersistCall& c, cudaStream_t st) {
    if (!c.plan.ok) return cudaErrorInvalidValue;
    const int D = c.dims.D;
    if (c.dims.mode == 2) {
        if (D <= 1024) return run_persist<2, 1>(c, st);
        if (D <= 2048) return run_persist<2, 2>(c, st);
        return run_persist<2, 4>(c, st);
    }
    if (D <= 1024) return run_persist<1, 1>(c, st);
    if (D <= 2048) return run_persist<1, 2>(c, st);
    return run_persist<1, 4>(c, st);
}

}  // namespace q8
