// The sparse mixture: top-k routing with the chunk's grouping, gate-up SwiGLU, down-and-combine.
//
// What it computes: forward_shim.rs module docs (a sparse mixture as a top-k router, a gate-up kernel and a
// down-and-combine kernel, its Q8_0 matrices dequantized inside the kernels that read them) and kernel_refusal (Moe
// arms: a softmax router whose kept weights are renormalized, SwiGLU experts, no biases); lane_link.rs, Link::prim Moe
// (k <= 32, experts <= 8192) and Link::class_launch MoeTokenSort (a chunk's choices grouped by expert, each expert's
// weights read once); lane/arena.rs, scratch (choices i, weights g, router logits rl, counts ec, offsets eo, lists el,
// hidden rows h and their quantized form hq/hs, weighed partials pa); qwen_emit docs, MoeWeights (stacked experts
// indexed by base offset e*dff / e*d).
//
// How (GB300 design): the expert products stream their weight rows exactly as the projection kernel does (one 256-bit
// load per 32-value block per lane, activations in registers).  Work items are (expert group, row-set, k-slice); a
// group is one expert and the choices routed to it, so a chunk reads each chosen expert's rows once.  Partial sums meet
// in workspace scratch; per-item arrival counters let the last arriver finish the item (slices summed in order, SwiGLU,
// the int8 epilogue of a 32-row block, or the gated combine over the row's k experts in choice order).
#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace q8 {
namespace {


// ==== top-k and grouping ==========================================================================================

constexpr int TOPK_THREADS = 256;  // a warp per row; the grid covers the rows
constexpr int TOPK_IDS_SMEM = 16384;  // choices staged in shared memory for the grouping (more: read from L2)

struct TopkParams {
    ExpertPrefetch xp;
    L2Prefetch pf;
    const float* logits;
    int R, E, K;
    int32_t* ids;
    float* gates;
    int32_t* counts;
    int32_t* offsets;
    int32_t* lists;
    int32_t* active;
    int* done;  // grid > 1 with a plan: arrivals of the CTAs (left zero); the last one groups
};

// One thread's prefetch of [p, p + n) into L2 (16-byte-aligned interior, 64 KB pieces).
__device__ __forceinline__ void prefetch_range(const void* p, size_t n) {
    const uintptr_t a = ((uintptr_t)p + 15) & ~uintptr_t(15);
    const uintptr_t e = ((uintptr_t)p + n) & ~uintptr_t(15);
    for (uintptr_t o = a; o < e; o += kPrefetchPiece) {
        const uintptr_t m = e - o < kPrefetchPiece ? e - o : kPrefetchPiece;
        l2_prefetch_piece((const char*)o, (unsigned)m);
    }
}

__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
    return be < 0 || v > bv || (v == bv && e < be);
}

// Exclusive scan of n ints in shared memory (in place), all threads of the CTA; returns the total.
__device__ int block_exclusive_scan(int* a, int n, int* tmp) {
    const int t = threadIdx.x, T = blockDim.x;
    const int per = (n + T - 1) / T;
    const int lo = t * per, hi = min(n, lo + per);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += a[i];
    // inclusive scan of the per-thread sums across the CTA
    const int lane = t & 31, wid = t >> 5;
    int v = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) tmp[wid] = v;
    __syncthreads();
    if (wid == 0) {
        int w = lane < (T >> 5) ? tmp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        tmp[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    int run = v - local + (wid > 0 ? tmp[wid - 1] : 0);
    const int total = tmp[(T >> 5) - 1];
    __syncthreads();
    for (int i = lo; i < hi; ++i) {
        const int x = a[i];
        a[i] = run;
        run += x;
    }
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(TOPK_THREADS) topk_kernel(const TopkParams p) {
    extern __shared__ int sm[];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    constexpr int NW = TOPK_THREADS / 32;
    issue_l2_prefetch(p.pf);
    griddep_wait();
    griddep_launch();
    for (int r = blockIdx.x * NW + wid; r < p.R; r += gridDim.x * NW) {
        const float* l = p.logits + (int64_t)r * p.E;
        // the row's logits in registers (up to 512 experts), else read from global memory each round
        constexpr int EPL = 16;
        float lr[EPL];
        const bool in_regs = p.E <= 32 * EPL;
        if (in_regs)
#pragma unroll
            for (int u = 0; u < EPL; ++u) {
                const int e = lane + 32 * u;
                lr[u] = e < p.E ? l[e] : -FLT_MAX;
            }
        float pv = FLT_MAX;
        int pi = -1;
        float kept = 0.f;  // lane j holds the j-th kept logit
        int kept_id = -1;
        for (int j = 0; j < p.K; ++j) {
            float bv = -FLT_MAX;
            int bi = -1;
            if (in_regs) {
#pragma unroll
                for (int u = 0; u < EPL; ++u) {
                    const int e = lane + 32 * u;
                    const float v = lr[u];
                    const bool eligible = e < p.E && (pi < 0 || v < pv || (v == pv && e > pi));
                    if (eligible && better(v, e, bv, bi)) {
                        bv = v;
                        bi = e;
                    }
                }
            } else {
                for (int e = lane; e < p.E; e += 32) {
                    const float v = l[e];
                    const bool eligible = pi < 0 || v < pv || (v == pv && e > pi);
                    if (eligible && better(v, e, bv, bi)) {
                        bv = v;
                        bi = e;
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (oi >= 0 && better(ov, oi, bv, bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (lane == j) {
                kept = bv;
                kept_id = bi;
            }
            pv = bv;
            pi = bi;
        }
        // gates: softmax over all experts renormalized over the kept ones = softmax over the kept logits
        const float m = __shfl_sync(0xffffffffu, kept, 0);
        const float pe = lane < p.K ? expf(kept - m) : 0.f;
        const float z = group_sum<32>(pe);
        if (lane < p.K) {
            p.ids[(int64_t)r * p.K + lane] = kept_id;
            p.gates[(int64_t)r * p.K + lane] = __fdiv_rn(pe, z);
        }
        // one row: the chosen experts' gate, up and down rows are fetched into L2 now, ahead of their kernels
        if (p.xp.gq && p.R == 1 && lane < p.K && kept_id >= 0 && kept_id < p.E) {
            const int64_t e = kept_id, dff = p.xp.dff, d = p.xp.d;
            prefetch_range(p.xp.gq + e * dff * d, (size_t)(dff * d));
            prefetch_range(p.xp.uq + e * dff * d, (size_t)(dff * d));
            prefetch_range(p.xp.dq + e * d * dff, (size_t)(d * dff));
            prefetch_range(p.xp.gs + e * dff * (d / 32), (size_t)(dff * (d / 32)) * 4);
            prefetch_range(p.xp.us + e * dff * (d / 32), (size_t)(dff * (d / 32)) * 4);
            prefetch_range(p.xp.ds + e * d * (dff / 32), (size_t)(d * (dff / 32)) * 4);
        }
    }
    if (!p.counts) return;
    if (gridDim.x > 1) {  // the last CTA to finish its rows groups them all
        __shared__ int last_s;
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) last_s = atomic_add_acq_rel_gpu(p.done, 1) == (int)gridDim.x - 1;
        __syncthreads();
        if (!last_s) return;
        if (threadIdx.x == 0) *p.done = 0;
    }
    __syncthreads();
    // grouping: counts, offsets, stable lists, active experts
    const int n = p.R * p.K;
    int* cnt = sm;                 // [E]
    int* flag = sm + p.E;          // [E]
    int* tmp = sm + 2 * p.E;       // [32]
    int* sid = sm + 2 * p.E + 32;  // [n] when n <= TOPK_IDS_SMEM
    const bool staged = n <= TOPK_IDS_SMEM;
    for (int e = threadIdx.x; e < p.E; e += TOPK_THREADS) cnt[e] = 0;
    if (staged)
        for (int c = threadIdx.x; c < n; c += TOPK_THREADS) sid[c] = __ldcg(p.ids + c);
    __syncthreads();
    for (int c = threadIdx.x; c < n; c += TOPK_THREADS) {
        const int e = staged ? sid[c] : __ldcg(p.ids + c);
        if (e >= 0 && e < p.E) atomicAdd(&cnt[e], 1);  // a row whose logits were all NaN chose no expert
    }
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += TOPK_THREADS) {
        p.counts[e] = cnt[e];
        flag[e] = cnt[e] > 0 ? 1 : 0;
    }
    __syncthreads();
    block_exclusive_scan(cnt, p.E, tmp);
    const int nactive = block_exclusive_scan(flag, p.E, tmp);
    for (int e = threadIdx.x; e < p.E; e += TOPK_THREADS) {
        p.offsets[e] = cnt[e];
        if (p.counts[e] > 0) p.active[1 + flag[e]] = e;
    }
    if (threadIdx.x == 0) {
        p.offsets[p.E] = cnt[p.E - 1] + p.counts[p.E - 1];
        p.active[0] = nactive;
    }
    __syncthreads();
    // stable scatter, choices in order: warp 0 takes 32 at a time; the lanes holding the same expert find each other
    // (match), the lowest of them advances the expert's cursor (cnt, now the offsets) past all of them
    if (wid == 0) {
        for (int c0 = 0; c0 < n; c0 += 32) {
            const int c = c0 + lane;
            int e = c < n ? (staged ? sid[c] : __ldcg(p.ids + c)) : -1;
            if (e < 0 || e >= p.E) e = -1;
            const unsigned same = __match_any_sync(0xffffffffu, e);
            if (e >= 0) {
                const int rank = __popc(same & ((1u << lane) - 1u));
                p.lists[cnt[e] + rank] = c;
            }
            __syncwarp();
            if (e >= 0 && (same & ((1u << lane) - 1u)) == 0) cnt[e] += __popc(same);
            __syncwarp();
        }
    }
}

// ==== the f32 router ================================================================================================

// A router of f32 values (lane_link.rs, Link::prim: Router::F32).  Warp e owns router row e and every activation row r:
// lane l multiplies columns 4l .. 4l+3 of each 128-column stripe in f32 and adds the stripe's partial into an f64
// accumulator; the warp's lanes are summed in f64.
__global__ void __launch_bounds__(256) router_f32_kernel(const float* __restrict__ w, int E, int d,
                                                         const float* __restrict__ x, int R, float* logits) {
    const int lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
    griddep_wait();
    griddep_launch();
    if (e >= E) return;
    const float* wr = w + (int64_t)e * d;
    for (int r = 0; r < R; ++r) {
        const float* xr = x + (int64_t)r * d;
        double acc = 0.0;
        for (int c = 4 * lane; c < d; c += 128) {
            const float4 wv = *reinterpret_cast<const float4*>(wr + c);
            const float4 xv = *reinterpret_cast<const float4*>(xr + c);
            const float part = fmaf(wv.w, xv.w, fmaf(wv.z, xv.z, fmaf(wv.y, xv.y, wv.x * xv.x)));
            acc += (double)part;
        }
        acc = group_sum<32>(acc);
        if (lane == 0) logits[(int64_t)r * E + e] = (float)acc;
    }
}

// h[i] = silu(g[i]) * u[i] (the shared expert's gated pair, as the expert kernels form it).
__global__ void __launch_bounds__(256) swiglu_kernel(const float* __restrict__ g, const float* __restrict__ u,
                                                     float* __restrict__ h, int64_t n) {
    griddep_wait();
    griddep_launch();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        h[i] = silu_f32(g[i]) * u[i];
}

// ==== expert products =============================================================================================

struct ExpertParams {
    int mode;
    const int8_t* q0;
    const float* s0;
    const int8_t* q1;
    const float* s1;
    int E, out_rows, k, nb;
    int R, K;
    const int32_t* ids;
    const float* gates;
    const int32_t* offsets;
    const int32_t* lists;
    const int32_t* active;
    const float* x;         // gate-up: [R][k]; down: h [R*K][k] f32
    const int8_t* xq;       // gate-up: [R][k]; down: hq [R*K][k]
    const int8_t* xl;       // mode 2: the low words beside xq
    const float* xs;
    float* h;               // gate-up out [R*K][out_rows]
    const float* residual;  // down
    float* y;               // down out [R][out_rows]
    float* expert_out;      // down out [R*K][out_rows]
    void* partial;          // down over a chunk: [R*K][out_rows] (f64 in mode 0, f32 in mode 1)
    int nrs;                // items per group (row tiles of out_rows)
    int mma_lo, mma_hi;     // groups of mma_lo..mma_hi choices are left to the tensor-core kernel (0: none)
    int xstage;             // gate-up, int8 modes: bytes of the chunk's activation rows staged in shared memory (0: none)
    L2Prefetch pf;
};

struct Group {
    int expert, c0, nc;
};

__device__ __forceinline__ int n_groups(const ExpertParams& p) { return p.active ? p.active[0] : p.K; }

__device__ __forceinline__ Group group_of(const ExpertParams& p, int a) {
    if (p.active) {
        const int e = p.active[1 + a];
        return Group{e, p.offsets[e], p.offsets[e + 1] - p.offsets[e]};
    }
    return Group{p.ids[a], a, 1};
}

__device__ __forceinline__ int choice_of(const ExpertParams& p, const Group& g, int i) {
    return p.active ? p.lists[g.c0 + i] : g.c0 + i;
}

// Gate-up: item (group a, row tile) — the tile's gate and up rows of expert e are loaded once into registers and
// multiplied by every choice routed to e: h[c][i] = silu(g . x_r) * (u . x_r), r the choice's token row.
template <int MODE, int LPR, int BPL, int RT>
__global__ void __launch_bounds__(Q8_THREADS, 1) gate_up_kernel(const ExpertParams p) {
    using T = typename AccType<MODE>::T;
    constexpr int RPW = 32 / LPR;
    constexpr int ROWS = RPW * RT;
    const int lane = threadIdx.x & 31, lg = lane % LPR, grp = lane / LPR;
    const int warp = blockIdx.x * Q8_WARPS + (threadIdx.x >> 5);
    const int W = gridDim.x * Q8_WARPS;
    int bidx[BPL];
    bool bval[BPL];
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        bidx[j] = lg + j * LPR;
        bval[j] = bidx[j] < p.nb;
    }
    issue_l2_prefetch(p.pf);
    griddep_wait();
    griddep_launch();
    // int8 mode, a chunk whose activation rows fit: they are staged in shared memory once, so a warp's turn to the
    // next row of its group reads shared memory rather than waiting on L2
    extern __shared__ __align__(16) unsigned char gsm[];
    const int8_t* xqb = p.xq;
    const int8_t* xlb = p.xl;
    const float* xsb = p.xs;
    if (MODE >= 1 && p.xstage) {
        const int64_t nq = (int64_t)p.R * p.k;  // a multiple of 32
        for (int64_t i = threadIdx.x; i < nq / 16; i += blockDim.x)
            reinterpret_cast<uint4*>(gsm)[i] = __ldcg(reinterpret_cast<const uint4*>(p.xq) + i);
        if (MODE == 2)  // the low words after the high words
            for (int64_t i = threadIdx.x; i < nq / 16; i += blockDim.x)
                reinterpret_cast<uint4*>(gsm + nq)[i] = __ldcg(reinterpret_cast<const uint4*>(p.xl) + i);
        float* sxs = reinterpret_cast<float*>(gsm + nq * (MODE == 2 ? 2 : 1));
        for (int64_t i = threadIdx.x; i < (int64_t)p.R * p.nb; i += blockDim.x) sxs[i] = __ldcg(p.xs + i);
        __syncthreads();
        xqb = reinterpret_cast<const int8_t*>(gsm);
        xlb = reinterpret_cast<const int8_t*>(gsm + nq);
        xsb = sxs;
    }
    const int items = n_groups(p) * p.nrs;
    XTile<MODE, BPL> x;
    int loaded = -1;
    for (int it = warp; it < items; it += W) {
        const int a = it / p.nrs, rs = it % p.nrs;
        const Group g = group_of(p, a);
        // an expert id outside [0, E) reads no weights and counts as an expert of zero weights
        const bool ev = g.expert >= 0 && g.expert < p.E;
        if (p.mma_lo && ev && g.nc >= p.mma_lo && g.nc <= p.mma_hi) continue;  // on the tensor cores
        const int i0 = rs * ROWS + grp * RT;
        const int nvalid = min(RT, p.out_rows - i0);
        const int64_t wrow = (int64_t)(ev ? g.expert : 0) * p.out_rows + i0;
        WTile<BPL, RT> tg, tu;
        load_tile<BPL, RT>(tg, p.q0, p.s0, wrow, ev ? nvalid : 0, p.k, p.nb, bidx, bval);
        load_tile<BPL, RT>(tu, p.q1, p.s1, wrow, ev ? nvalid : 0, p.k, p.nb, bidx, bval);
        for (int ci = 0; ci < g.nc; ++ci) {
            const int c = choice_of(p, g, ci);
            const int xrow = c / p.K;
            if (xrow != loaded) {
                load_x<MODE, BPL>(x, p.x + (int64_t)xrow * p.k, xqb + (int64_t)xrow * p.k, xlb + (int64_t)xrow * p.k,
                                  xsb + (int64_t)xrow * p.nb, bidx, bval);
                loaded = xrow;
            }
#pragma unroll
            for (int i = 0; i < RT; ++i) {
                const T gv = group_sum<LPR>(tile_row_dot<MODE, BPL, RT>(tg, i, x));
                const T uv = group_sum<LPR>(tile_row_dot<MODE, BPL, RT>(tu, i, x));
                if (lg == 0 && i < nvalid) p.h[(int64_t)c * p.out_rows + i0 + i] = silu_f32((float)gv) * (float)uv;
            }
        }
    }
}

constexpr int DOWN_SMEM_MAX = 96 * 1024;

// Down-and-combine for one token row: the CTA first stages the k hidden rows in shared memory (quantized there in the
// int8 mode when given f32).  A warp owns one output row o; its 32/LPR lane groups take the kept experts round-robin
// (group gi: experts gi, gi + 32/LPR, ...), so every expert's row o is loaded at once across the warp, and lane 0
// gathers the k dot products and forms y = residual + sum_j g_j * (Wd[e_j] . h_j) in choice order.
template <int MODE, int LPR, int BPL>
__global__ void __launch_bounds__(Q8_THREADS, 1) down_one_kernel(const ExpertParams p) {
    using T = typename AccType<MODE>::T;
    extern __shared__ __align__(16) unsigned char dsm[];
    constexpr int NG = 32 / LPR;   // lane groups = experts in flight per pass
    const int lane = threadIdx.x & 31, lg = lane % LPR, gi = lane / LPR, wid = threadIdx.x >> 5;
    const int warp = blockIdx.x * Q8_WARPS + wid;
    const int W = gridDim.x * Q8_WARPS;
    const int K = p.K, kk = p.k;
    int bidx[BPL];
    bool bval[BPL];
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        bidx[j] = lg + j * LPR;
        bval[j] = bidx[j] < p.nb;
    }
    // the routing (ids, gates) was written two launches back, before the previous kernel passed its own wait
    const int npass = (K + NG - 1) / NG;
    issue_l2_prefetch(p.pf);
    griddep_wait();
    griddep_launch();
    float* hf = reinterpret_cast<float*>(dsm);                              // [K][kk] f32 staging
    int8_t* hq = reinterpret_cast<int8_t*>(dsm + (size_t)K * kk * 4);       // [K][kk] words (int8 modes)
    int8_t* hl = reinterpret_cast<int8_t*>(dsm + (size_t)K * kk * 5);       // [K][kk] low words (mode 2)
    float* hs = reinterpret_cast<float*>(dsm + (size_t)K * kk * (MODE == 2 ? 6 : 5));  // [K][kk/32] scales
    if (MODE == 0 || p.x) {
        for (int i = threadIdx.x; i < K * kk / 4; i += Q8_THREADS)
            reinterpret_cast<float4*>(hf)[i] = __ldcg(reinterpret_cast<const float4*>(p.x) + i);
        __syncthreads();
        if (MODE >= 1)
            for (int b = wid; b < K * kk / 32; b += Q8_WARPS) {
                float dsc;
                if (MODE == 2) {
                    int8_t lv;
                    hq[b * 32 + lane] = quantize2_lane(hf[b * 32 + lane], dsc, lv);
                    hl[b * 32 + lane] = lv;
                } else {
                    hq[b * 32 + lane] = quantize_lane(hf[b * 32 + lane], dsc);
                }
                if (lane == 0) hs[b] = dsc;
            }
    } else {
        for (int i = threadIdx.x; i < K * kk / 16; i += Q8_THREADS)
            reinterpret_cast<uint4*>(hq)[i] = __ldcg(reinterpret_cast<const uint4*>(p.xq) + i);
        if (MODE == 2)
            for (int i = threadIdx.x; i < K * kk / 16; i += Q8_THREADS)
                reinterpret_cast<uint4*>(hl)[i] = __ldcg(reinterpret_cast<const uint4*>(p.xl) + i);
        for (int i = threadIdx.x; i < K * kk / 32; i += Q8_THREADS) hs[i] = __ldcg(p.xs + i);
    }
    __syncthreads();
    for (int o = warp; o < p.out_rows; o += W) {
        T acc = 0;
        // passes of NG experts (expert j = m*NG + gi), two passes' loads in flight at a time
        for (int m0 = 0; m0 < npass; m0 += 2) {
            WTile<BPL, 1> t[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int j = (m0 + u) * NG + gi;
                const int e = j < K ? __ldg(p.ids + j) : -1;
                const bool ev = e >= 0 && e < p.E;
                load_tile<BPL, 1>(t[u], p.q0, p.s0, (int64_t)(ev ? e : 0) * p.out_rows + o, ev ? 1 : 0, kk, p.nb,
                                  bidx, bval);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int m = m0 + u;
                if (m >= npass) break;
                const int j = m * NG + gi;
                const int jj = j < K ? j : 0;
                XTile<MODE, BPL> x;
                load_x<MODE, BPL>(x, hf + (int64_t)jj * kk, hq + (int64_t)jj * kk, hl + (int64_t)jj * kk,
                                  hs + (int64_t)jj * p.nb, bidx, bval);
                const T mine = group_sum<LPR>(tile_row_dot<MODE, BPL, 1>(t[u], 0, x));
                // lane 0 adds this pass's experts in choice order
                for (int g = 0; g < NG; ++g) {
                    const T ej = __shfl_sync(0xffffffffu, mine, g * LPR);
                    const int jg = m * NG + g;
                    if (lane == 0 && jg < K) {
                        if (p.expert_out) p.expert_out[(int64_t)jg * p.out_rows + o] = (float)ej;
                        const float gj = __ldg(p.gates + jg);
                        acc = (MODE == 0) ? (T)fma((double)gj, (double)ej, (double)acc)
                                          : (T)fmaf(gj, (float)ej, (float)acc);
                    }
                }
            }
        }
        if (lane == 0) {
            float v = (float)acc;
            if (p.residual) v = p.residual[o] + v;
            p.y[o] = v;
        }
    }
}

// Down over a chunk: item (group a, row tile) — expert e's tile is loaded once and multiplied by every choice routed
// to it; each choice's unweighted output goes to scratch for the combine.
template <int MODE, int LPR, int BPL, int RT>
__global__ void __launch_bounds__(Q8_THREADS, 1) down_group_kernel(const ExpertParams p) {
    using T = typename AccType<MODE>::T;
    constexpr int RPW = 32 / LPR;
    constexpr int ROWS = RPW * RT;
    const int lane = threadIdx.x & 31, lg = lane % LPR, grp = lane / LPR;
    const int warp = blockIdx.x * Q8_WARPS + (threadIdx.x >> 5);
    const int W = gridDim.x * Q8_WARPS;
    int bidx[BPL];
    bool bval[BPL];
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        bidx[j] = lg + j * LPR;
        bval[j] = bidx[j] < p.nb;
    }
    griddep_wait();
    griddep_launch();
    const int items = n_groups(p) * p.nrs;
    T* part = reinterpret_cast<T*>(p.partial);
    for (int it = warp; it < items; it += W) {
        const int a = it / p.nrs, rs = it % p.nrs;
        const Group g = group_of(p, a);
        const bool ev = g.expert >= 0 && g.expert < p.E;
        if (p.mma_lo && ev && g.nc >= p.mma_lo && g.nc <= p.mma_hi) continue;  // on the tensor cores
        const int o0 = rs * ROWS + grp * RT;
        const int nvalid = min(RT, p.out_rows - o0);
        WTile<BPL, RT> t;
        load_tile<BPL, RT>(t, p.q0, p.s0, (int64_t)(ev ? g.expert : 0) * p.out_rows + o0, ev ? nvalid : 0, p.k, p.nb,
                           bidx, bval);
        for (int ci = 0; ci < g.nc; ++ci) {
            const int c = choice_of(p, g, ci);
            XTile<MODE, BPL> x;
            load_x<MODE, BPL>(x, p.x + (int64_t)c * p.k, p.xq + (int64_t)c * p.k, p.xl + (int64_t)c * p.k,
                              p.xs + (int64_t)c * p.nb, bidx, bval);
#pragma unroll
            for (int i = 0; i < RT; ++i) {
                const T e = group_sum<LPR>(tile_row_dot<MODE, BPL, RT>(t, i, x));
                if (lg == 0 && i < nvalid) part[(int64_t)c * p.out_rows + o0 + i] = e;
            }
        }
    }
}

// y[r][o] = residual[r][o] + sum_j g[r][j] * part[r*K + j][o], the experts in choice order.
template <int MODE>
__global__ void __launch_bounds__(256) combine_kernel(const ExpertParams p) {
    using T = typename AccType<MODE>::T;
    griddep_wait();
    griddep_launch();
    const T* part = reinterpret_cast<const T*>(p.partial);
    const int64_t n = (int64_t)p.R * p.out_rows;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / p.out_rows, o = i % p.out_rows;
        T acc = 0;
        for (int j = 0; j < p.K; ++j) {
            const int64_t c = r * p.K + j;
            const T e = part[c * p.out_rows + o];
            if (p.expert_out) p.expert_out[c * p.out_rows + o] = (float)e;
            acc = (MODE == 0) ? (T)fma((double)p.gates[c], (double)e, (double)acc)
                              : (T)fmaf(p.gates[c], (float)e, (float)acc);
        }
        float v = (float)acc;
        if (p.residual) v = p.residual[i] + v;
        p.y[i] = v;
    }
}

struct EPlan {
    int lpr, bpl, rt;
    int rows() const { return 32 / lpr * rt; }
};

// One slice over k, every lane busy; about target_loads 32-byte loads in flight per lane.
EPlan eplan(int mode, int nb, int target_loads) {
    const int bpl_max = (mode == 0) ? 3 : 4;
    EPlan best{32, 1, 1};
    int bestS = 1 << 30;
    double best_util = -1.0;
    for (int lpr : {32, 16, 8}) {
        for (int bpl = 1; bpl <= bpl_max; ++bpl) {
            const int sb = lpr * bpl;
            const int S = (nb + sb - 1) / sb;
            const double util = (double)nb / (double)(S * sb);
            if (S < bestS || (S == bestS && util > best_util + 1e-9)) {
                bestS = S;
                best_util = util;
                best = EPlan{lpr, bpl, 1};
            }
        }
    }
    const int rt = target_loads / best.bpl;
    best.rt = rt >= 4 ? 4 : (rt >= 2 ? 2 : 1);
    if (best.bpl > 2 && best.rt > 2) best.rt = 2;
    return best;
}

ExpertParams make_params(const ExpertCall& c, const EPlan& pl) {
    ExpertParams p = {};
    p.mode = c.mode;
    p.q0 = c.q0;
    p.s0 = c.s0;
    p.q1 = c.q1;
    p.s1 = c.s1;
    p.E = (int)c.E;
    p.out_rows = (int)c.out_rows;
    p.k = (int)c.k;
    p.nb = (int)(c.k / 32);
    p.R = (int)c.R;
    p.K = c.K;
    p.ids = c.ids;
    p.gates = c.gates;
    p.offsets = c.plan.offsets;
    p.lists = c.plan.lists;
    p.active = c.plan.active;
    p.x = c.x;
    p.xq = c.xq;
    p.xl = c.xl;
    p.xs = c.xs;
    p.h = c.h;
    p.residual = c.residual;
    p.y = c.y;
    p.expert_out = c.expert_out;
    p.nrs = (int)((c.out_rows + pl.rows() - 1) / pl.rows());
    p.pf = c.pf;
    return p;
}


int max_groups(const ExpertCall& c) {
    const int64_t choices = c.R * c.K;
    return (int)(choices < c.E ? choices : c.E);
}

size_t down_one_smem(const ExpertCall& c) {
    return (size_t)c.K * c.k * 4 + (c.mode >= 1 ? (size_t)c.K * c.k * c.mode + (size_t)c.K * c.k / 32 * 4 : 0);
}

#define Q8_EXPERT_ONE(KERNEL, MODE, L, B, R)                                                               \
    if (pl.lpr == L && pl.bpl == B && pl.rt == R) {                                                        \
        auto kern = KERNEL<MODE, L, B, R>;                                                                 \
        if (p.xstage > 48 * 1024) {                                                                        \
            const cudaError_t ae =                                                                         \
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p.xstage);         \
            if (ae != cudaSuccess) return ae;                                                              \
        }                                                                                                  \
        return launch(kern, dim3(persistent_grid(kern, p.xstage, warps)), dim3(Q8_THREADS), (size_t)p.xstage, \
                      st, c.pdl, p);                                                                       \
    }
#define Q8_EXPERT_LPR(KERNEL, MODE, L)                                                                     \
    Q8_EXPERT_ONE(KERNEL, MODE, L, 1, 1) Q8_EXPERT_ONE(KERNEL, MODE, L, 1, 2) Q8_EXPERT_ONE(KERNEL, MODE, L, 1, 4) \
    Q8_EXPERT_ONE(KERNEL, MODE, L, 2, 1) Q8_EXPERT_ONE(KERNEL, MODE, L, 2, 2) Q8_EXPERT_ONE(KERNEL, MODE, L, 3, 1) \
    if (MODE >= 1) {                                                                                       \
        Q8_EXPERT_ONE(KERNEL, MODE, L, 2, 4) Q8_EXPERT_ONE(KERNEL, MODE, L, 3, 2)                          \
        Q8_EXPERT_ONE(KERNEL, MODE, L, 4, 1) Q8_EXPERT_ONE(KERNEL, MODE, L, 4, 2)                          \
    }
#define Q8_EXPERT_DISPATCH(KERNEL, MODE)                                                                   \
    do {                                                                                                   \
        Q8_EXPERT_LPR(KERNEL, MODE, 32) Q8_EXPERT_LPR(KERNEL, MODE, 16) Q8_EXPERT_LPR(KERNEL, MODE, 8)     \
    } while (0)

template <int MODE>
cudaError_t run_gate_up(const ExpertCall& c, const EPlan& pl, const ExpertParams& p, int64_t warps, cudaStream_t st) {
    Q8_EXPERT_DISPATCH(gate_up_kernel, MODE);
    return cudaErrorInvalidConfiguration;
}

template <int MODE>
cudaError_t run_down_group(const ExpertCall& c, const EPlan& pl, const ExpertParams& p, int64_t warps, cudaStream_t st) {
    Q8_EXPERT_DISPATCH(down_group_kernel, MODE);
    return cudaErrorInvalidConfiguration;
}

template <int MODE, int L, int B>
cudaError_t run_down_one(const ExpertParams& p, int64_t warps, size_t smem, cudaStream_t st, int pdl) {
    auto kern = down_one_kernel<MODE, L, B>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DOWN_SMEM_MAX);
    if (e != cudaSuccess) return e;
    return launch(kern, dim3(persistent_grid(kern, smem, warps)), dim3(Q8_THREADS), smem, st, pdl, p);
}

template <int MODE>
cudaError_t dispatch_down_one(const EPlan& pl, const ExpertParams& p, int64_t grid, size_t smem, cudaStream_t st, int pdl) {
    if (pl.lpr == 32 && pl.bpl == 1) return run_down_one<MODE, 32, 1>(p, grid, smem, st, pdl);
    if (pl.lpr == 32 && pl.bpl == 2) return run_down_one<MODE, 32, 2>(p, grid, smem, st, pdl);
    if (pl.lpr == 32 && pl.bpl == 3) return run_down_one<MODE, 32, 3>(p, grid, smem, st, pdl);
    if (pl.lpr == 16 && pl.bpl == 1) return run_down_one<MODE, 16, 1>(p, grid, smem, st, pdl);
    if (pl.lpr == 16 && pl.bpl == 2) return run_down_one<MODE, 16, 2>(p, grid, smem, st, pdl);
    if (pl.lpr == 16 && pl.bpl == 3) return run_down_one<MODE, 16, 3>(p, grid, smem, st, pdl);
    if (pl.lpr == 8 && pl.bpl == 1) return run_down_one<MODE, 8, 1>(p, grid, smem, st, pdl);
    if (pl.lpr == 8 && pl.bpl == 2) return run_down_one<MODE, 8, 2>(p, grid, smem, st, pdl);
    if (pl.lpr == 8 && pl.bpl == 3) return run_down_one<MODE, 8, 3>(p, grid, smem, st, pdl);
    if (MODE >= 1) {
        if (pl.lpr == 32 && pl.bpl == 4) return run_down_one<MODE, 32, 4>(p, grid, smem, st, pdl);
        if (pl.lpr == 16 && pl.bpl == 4) return run_down_one<MODE, 16, 4>(p, grid, smem, st, pdl);
        if (pl.lpr == 8 && pl.bpl == 4) return run_down_one<MODE, 8, 4>(p, grid, smem, st, pdl);
    }
    return cudaErrorInvalidConfiguration;
}

}  // namespace

cudaError_t launch_topk(const TopkCall& c, cudaStream_t st) {
    TopkParams p = {c.xp, c.pf, c.logits, (int)c.R, (int)c.E, c.K, c.ids, c.gates,
                    c.plan.counts, c.plan.offsets, c.plan.lists, c.plan.active, c.done};
    constexpr int NW = TOPK_THREADS / 32;
    int64_t grid = (c.R + NW - 1) / NW;
    if (grid > device_info().sms) grid = device_info().sms;
    if (grid < 1) grid = 1;
    if (c.plan.counts && grid > 1 && !c.done) grid = 1;  // no arrival counter: one CTA takes every row
    const int64_t n = c.R * c.K;
    const size_t smem = c.plan.counts ? (size_t)(2 * c.E + 32 + (n <= TOPK_IDS_SMEM ? n : 0)) * sizeof(int) : 0;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch(topk_kernel, dim3((unsigned)grid), dim3(TOPK_THREADS), smem, st, c.pdl, p);
}

bool experts_supported(int mode, int64_t k) { return k / 32 <= 32 * ((mode == 0) ? 3 : 4); }

void gate_up_scratch(const ExpertCall& c, size_t* bytes, size_t* counters) {
    *bytes = 0;
    *counters = c.hq_out ? (size_t)(c.R * c.K * (c.out_rows / 32)) : 0;
}

cudaError_t launch_down_routed(const ExpertCall& c, Carve& ws, cudaStream_t st);

void down_scratch(const ExpertCall& c, size_t* bytes, size_t* counters) {
    const bool one = down_row_supported(c) ||
                     (c.R == 1 && !c.plan.active && c.K <= 32 && down_one_smem(c) <= (size_t)DOWN_SMEM_MAX);
    *bytes = one ? 0 : (size_t)c.R * c.K * c.out_rows * (c.mode == 0 ? 8 : 4);
    *counters = 0;
}

cudaError_t launch_router_f32(const float* w, int64_t E, int64_t d, const float* x, int64_t R, float* logits,
                              int pdl, cudaStream_t st) {
    return launch(router_f32_kernel, dim3((unsigned)((E + 7) / 8)), dim3(256), 0, st, pdl, w, (int)E, (int)d, x,
                  (int)R, logits);
}

namespace {

// The shared expert's gated pair for the forms that do not fuse it: one two-segment projection (gate and up rows of
// every activation row), then h = silu(g) * u into the hidden rows after the routed ones.
cudaError_t shared_gate_up(const ExpertCall& c, Carve& ws, cudaStream_t st) {
    const int64_t n = c.R * c.sdff;
    float* g = ws.take<float>((size_t)n);
    float* u = ws.take<float>((size_t)n);
    if (ws.overflow) return cudaErrorMemoryAllocation;
    GemvCall pc;
    pc.mode = c.mode;
    pc.k = c.k;
    pc.nseg = 2;
    pc.seg[0] = GemvSeg{c.sq0, c.ss0, c.sdff, g, nullptr};
    pc.seg[1] = GemvSeg{c.sq1, c.ss1, c.sdff, u, nullptr};
    pc.x = c.x;
    pc.xq = c.xq;
    pc.xl = c.xl;
    pc.xs = c.xs;
    pc.R = c.R;
    pc.err = c.err;
    pc.pdl = c.pdl;
    cudaError_t e = launch_gemv(pc, ws, st);
    if (e != cudaSuccess) return e;
    int grid = (int)((n + 255) / 256);
    if (grid > device_info().sms * 4) grid = device_info().sms * 4;
    return launch(swiglu_kernel, dim3(grid), dim3(256), 0, st, c.pdl, (const float*)g, (const float*)u,
                  c.h + c.R * c.K * c.out_rows, n);
}

// The shared expert's down product for the forms that do not fuse it, added onto y (which already holds the residual
// and the routed experts' weighted sum): y = y + Wd_s . h_s.
cudaError_t shared_down(const ExpertCall& c, Carve& ws, cudaStream_t st) {
    const int64_t off = c.R * c.K * c.k;  // the shared hidden rows follow the routed ones
    GemvCall pc;
    pc.mode = c.mode;
    pc.k = c.sdff;
    pc.seg[0] = GemvSeg{c.sq0, c.ss0, c.out_rows, c.y, c.y};
    pc.R = c.R;
    pc.err = c.err;
    pc.pdl = c.pdl;
    if (c.mode == 0) {
        pc.x = c.x + off;
    } else if (c.xq) {
        pc.xq = c.xq + off;
        pc.xl = c.xl ? c.xl + off : nullptr;
        pc.xs = c.xs + off / 32;
    } else {  // f32 hidden rows in an int8 mode: the shared rows quantized here
        const int64_t n = c.R * c.sdff;
        int8_t* q = ws.take<int8_t>((size_t)n);
        int8_t* l = c.mode == 2 ? ws.take<int8_t>((size_t)n) : nullptr;
        float* s = ws.take<float>((size_t)(n / 32));
        if (ws.overflow) return cudaErrorMemoryAllocation;
        cudaError_t e = launch_quantize(c.x + off, n, q, s, st, l);
        if (e != cudaSuccess) return e;
        pc.xq = q;
        pc.xl = l;
        pc.xs = s;
    }
    return launch_gemv(pc, ws, st);
}

}  // namespace

namespace {

// The grouped tensor-core launch and the CUDA-core launch of a chunk read the same routing and write disjoint rows, so
// with plain launches the former runs on a side stream beside the latter: forked from `st` by an event, joined back
// by another.  One side stream and two events per thread and device, made on first use and kept for the thread's
// life.
struct Side {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

Side* side_stream() {
    constexpr int kDevices = 16;
    thread_local Side sides[kDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) return nullptr;
    Side& sd = sides[dev];
    if (!sd.s) {
        if (cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            sd = Side{};
            return nullptr;
        }
    }
    return &sd;
}

// Forks the side stream off `st`: work launched on the returned stream starts after what `st` holds so far.  Without
// a side stream (or if the fork fails), and while `st` is being captured into a graph, the work goes on `st` itself:
// measured in a replayed graph of eight uncorrelated 64-row chunks, the forked branches made a chunk 279 us against
// 207 us in order, while plain launches gain (a 64-row prefill chunk 21.1 ms against 23.2 ms).
cudaStream_t fork_side(cudaStream_t st, Side** used) {
    *used = nullptr;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return st;
    }
    Side* sd = side_stream();
    if (!sd || cudaEventRecord(sd->fork, st) != cudaSuccess || cudaStreamWaitEvent(sd->s, sd->fork, 0) != cudaSuccess) {
        cudaGetLastError();
        return st;
    }
    *used = sd;
    return sd->s;
}

// Joins the side stream back into `st`: what `st` runs next waits for the side stream's work.
cudaError_t join_side(cudaStream_t st, Side* sd) {
    if (!sd) return cudaSuccess;
    cudaError_t e = cudaEventRecord(sd->join, sd->s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, sd->join, 0);
    return e;
}

}  // namespace

cudaError_t launch_gate_up(const ExpertCall& c, Carve& ws, cudaStream_t st) {
    if (gate_row_supported(c)) return launch_gate_row(c, ws, st);  // the shared expert's rows are items of the kernel
    if (c.hq_out) return cudaErrorInvalidConfiguration;  // the int8 epilogue exists in the one-row kernel only
    // gate and up tiles are both in flight: about four (f32) or eight (int8) 32-byte loads per lane in all
    const EPlan pl = eplan(c.mode, (int)(c.k / 32), c.mode == 0 ? 2 : 4);
    ExpertParams p = make_params(c, pl);
    const bool mma = moe_mma_grouped(c);
    if (mma) {
        p.mma_lo = moe_mma_min_rows();
        p.mma_hi = moe_mma_max_rows();
    }
    const int64_t warps = (int64_t)max_groups(c) * p.nrs;
    const int64_t xbytes = c.R * c.k * c.mode + c.R * (c.k / 32) * 4;
    if (c.mode >= 1 && c.R > 1 && xbytes <= 96 * 1024 && (uintptr_t)c.xq % 16 == 0 &&
        (c.mode == 1 || (uintptr_t)c.xl % 16 == 0))
        p.xstage = (int)xbytes;
    Side* sd = nullptr;
    cudaError_t e = cudaSuccess;
    if (mma) {  // the groups of moe_mma_min_rows() choices or more, beside the CUDA-core launch
        ExpertCall cm = c;
        cm.pdl = 0;
        e = launch_moe_mma(cm, c.h, max_groups(c), ws, fork_side(st, &sd));
    }
    if (e == cudaSuccess)
        e = c.mode == 0 ? run_gate_up<0>(c, pl, p, warps, st)
          : c.mode == 1 ? run_gate_up<1>(c, pl, p, warps, st) : run_gate_up<2>(c, pl, p, warps, st);
    const cudaError_t ej = join_side(st, sd);
    if (e == cudaSuccess) e = ej;
    if (e == cudaSuccess && c.sdff) e = shared_gate_up(c, ws, st);
    return e;
}

cudaError_t launch_down_combine(const ExpertCall& c, Carve& ws, cudaStream_t st) {
    if (down_row_supported(c)) return launch_down_row(c, st);  // the shared expert's blocks are pairs of the kernel
    cudaError_t e = launch_down_routed(c, ws, st);
    if (e == cudaSuccess && c.sdff) e = shared_down(c, ws, st);
    return e;
}

cudaError_t launch_down_routed(const ExpertCall& c, Carve& ws, cudaStream_t st) {
    const int nb = (int)(c.k / 32);
    if (c.R == 1 && !c.plan.active && c.K <= 32 && down_one_smem(c) <= (size_t)DOWN_SMEM_MAX) {
        // one token: a warp per output row, its lane groups over the kept experts
        EPlan pl = eplan(c.mode, nb, 4);
        pl.rt = 1;
        ExpertParams p = make_params(c, pl);
        const int64_t grid = c.out_rows;
        const size_t smem = down_one_smem(c);
        return c.mode == 0 ? dispatch_down_one<0>(pl, p, grid, smem, st, c.pdl)
             : c.mode == 1 ? dispatch_down_one<1>(pl, p, grid, smem, st, c.pdl)
                           : dispatch_down_one<2>(pl, p, grid, smem, st, c.pdl);
    }
    // a chunk (or one row through a plan): grouped product into scratch, then the ordered combine
    const EPlan pl = eplan(c.mode, nb, c.mode == 0 ? 4 : 8);
    ExpertParams p = make_params(c, pl);
    p.partial = ws.take<char>((size_t)c.R * c.K * c.out_rows * (c.mode == 0 ? 8 : 4));
    if (ws.overflow) return cudaErrorMemoryAllocation;
    const bool mma = moe_mma_grouped(c);
    if (mma) {
        p.mma_lo = moe_mma_min_rows();
        p.mma_hi = moe_mma_max_rows();
    }
    const int64_t warps = (int64_t)max_groups(c) * p.nrs;
    Side* sd = nullptr;
    cudaError_t e = cudaSuccess;
    if (mma) {  // the groups of moe_mma_min_rows() choices or more, beside the CUDA-core launch
        ExpertCall cm = c;
        cm.pdl = 0;
        e = launch_moe_mma(cm, reinterpret_cast<float*>(p.partial), max_groups(c), ws, fork_side(st, &sd));
    }
    if (e == cudaSuccess)
        e = c.mode == 0 ? run_down_group<0>(c, pl, p, warps, st)
          : c.mode == 1 ? run_down_group<1>(c, pl, p, warps, st) : run_down_group<2>(c, pl, p, warps, st);
    const cudaError_t ej = join_side(st, sd);
    if (e == cudaSuccess) e = ej;
    if (e != cudaSuccess) return e;
    const int64_t n = c.R * c.out_rows;
    int cg = (int)((n + 255) / 256);
    if (cg > device_info().sms * 4) cg = device_info().sms * 4;
    return c.mode == 0 ? launch(combine_kernel<0>, dim3(cg), dim3(256), 0, st, c.pdl, p)
                       : launch(combine_kernel<1>, dim3(cg), dim3(256), 0, st, c.pdl, p);  // f32 sums in modes 1, 2
}

}  // namespace q8
