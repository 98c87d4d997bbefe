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

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

// ==== top-k and grouping ==========================================================================================

constexpr int TOPK_THREADS = 512;

struct TopkParams {
    const float* logits;
    int R, E, K;
    int32_t* ids;
    float* gates;
    int32_t* counts;
    int32_t* offsets;
    int32_t* lists;
    int32_t* active;
};

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
    griddep_wait();
    for (int r = wid; r < p.R; r += NW) {
        const float* l = p.logits + (int64_t)r * p.E;
        float pv = FLT_MAX;
        int pi = -1;
        float kept = 0.f;  // lane j holds the j-th kept logit
        int kept_id = -1;
        for (int j = 0; j < p.K; ++j) {
            float bv = -FLT_MAX;
            int bi = -1;
            for (int e = lane; e < p.E; e += 32) {
                const float v = l[e];
                const bool eligible = pi < 0 || v < pv || (v == pv && e > pi);
                if (eligible && better(v, e, bv, bi)) {
                    bv = v;
                    bi = e;
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
    }
    if (!p.counts) return;
    __syncthreads();
    // grouping: counts, offsets, stable lists, active experts
    int* cnt = sm;                 // [E]
    int* flag = sm + p.E;          // [E]
    int* tmp = sm + 2 * p.E;       // [32]
    const int n = p.R * p.K;
    for (int e = threadIdx.x; e < p.E; e += TOPK_THREADS) cnt[e] = 0;
    __syncthreads();
    for (int c = threadIdx.x; c < n; c += TOPK_THREADS) {
        const int e = p.ids[c];
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
    for (int c = threadIdx.x; c < n; c += TOPK_THREADS) {
        const int e = p.ids[c];
        if (e < 0 || e >= p.E) continue;
        int rank = 0;
        for (int c2 = 0; c2 < c; ++c2) rank += (p.ids[c2] == e);
        p.lists[cnt[e] + rank] = c;
    }
    griddep_launch();
}

// ==== expert products =============================================================================================

template <int MODE>
struct AccT;
template <>
struct AccT<0> {
    using T = double;
};
template <>
struct AccT<1> {
    using T = float;
};

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
    const float* x;
    const int8_t* xq;
    const float* xs;
    float* h;
    int8_t* hq;
    float* hs;
    const float* residual;
    float* y;
    float* expert_out;
    int S, nrs;
    void* partial;
    int* cnt_slice;   // gate-up: [R*K][nrs]
    int* cnt_quant;   // gate-up: [R*K][out_rows/32]
    int* cnt_row;     // down: [R][nrs]
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

// Loads one activation row's blocks for this lane.
template <int MODE, int BPL>
__device__ __forceinline__ void load_x(const float* x, const int8_t* xq, const float* xs, int64_t row, int k, int nb,
                                       const int (&bidx)[BPL], const bool (&bval)[BPL], float* xf,
                                       uint32_t (&xw)[MODE == 1 ? BPL : 1][8], float (&xsc)[BPL]) {
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        if (MODE == 0) {
            const float4* xp = reinterpret_cast<const float4*>(x + row * k + bidx[j] * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 v = bval[j] ? __ldcg(xp + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                xf[j * 32 + 4 * i + 0] = v.x;
                xf[j * 32 + 4 * i + 1] = v.y;
                xf[j * 32 + 4 * i + 2] = v.z;
                xf[j * 32 + 4 * i + 3] = v.w;
            }
            xsc[j] = 0.f;
        } else {
            if (bval[j]) {
                const uint4* xp = reinterpret_cast<const uint4*>(xq + row * k + bidx[j] * 32);
                const uint4 a = __ldcg(xp), b = __ldcg(xp + 1);
                xw[j][0] = a.x; xw[j][1] = a.y; xw[j][2] = a.z; xw[j][3] = a.w;
                xw[j][4] = b.x; xw[j][5] = b.y; xw[j][6] = b.z; xw[j][7] = b.w;
                xsc[j] = __ldcg(xs + row * nb + bidx[j]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) xw[j][i] = 0u;
                xsc[j] = 0.f;
            }
        }
    }
}

template <int MODE, int BPL>
__device__ __forceinline__ void load_w(const int8_t* q, const float* s, int64_t row, bool rv, int k, int nb,
                                       const int (&bidx)[BPL], const bool (&bval)[BPL], uint32_t (&w)[BPL][8],
                                       float (&sc)[BPL]) {
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        if (rv && bval[j]) {
            ld_block_stream(q + row * k + bidx[j] * 32, w[j]);
            sc[j] = ld_scale_stream(s + row * nb + bidx[j]);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) w[j][i] = 0u;
            sc[j] = 0.f;
        }
    }
}

template <int MODE, int BPL>
__device__ __forceinline__ typename AccT<MODE>::T dot(const uint32_t (&w)[BPL][8], const float (&sc)[BPL],
                                                      const float* xf, const uint32_t (&xw)[MODE == 1 ? BPL : 1][8],
                                                      const float (&xsc)[BPL]) {
    typename AccT<MODE>::T acc = 0;
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        if (MODE == 0) {
            const float ps = block_dot_f32(w[j], xf + j * 32);
            acc = fma((double)sc[j], (double)ps, (double)acc);
        } else {
            const int D = block_dot_i8(w[j], xw[j]);
            acc = fmaf(sc[j] * xsc[j], (float)D, (float)acc);
        }
    }
    return acc;
}

// After h[c][i0 .. i0+rows) is stored: count those rows into their 32-row block; the warp completing a block
// quantizes it (the int8 epilogue of the gate-up kernel).
template <int RPW>
__device__ __forceinline__ void quant_arrive(const ExpertParams& p, int c, int i0, int rows) {
    const int lane = threadIdx.x & 31;
    const int qb = i0 / 32;
    int* cnt = p.cnt_quant + (int64_t)c * (p.out_rows / 32) + qb;
    __threadfence();
    __syncwarp();
    int old = 0;
    if (lane == 0) old = atomicAdd(cnt, rows);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old + rows == 32) {
        __threadfence();
        const int64_t base = (int64_t)c * p.out_rows + qb * 32;
        const float v = __ldcg(p.h + base + lane);
        float d;
        const int8_t qv = quantize_lane(v, d);
        p.hq[base + lane] = qv;
        if (lane == 0) {
            p.hs[base / 32] = d;
            *cnt = 0;
        }
    }
}

// Gate-up: item (group a, row-set rs) on slice `slice`; rows i of expert e: h = silu(g . x) * (u . x).
template <int MODE, int LPR, int BPL>
__global__ void __launch_bounds__(Q8_THREADS, 2) gate_up_kernel(const ExpertParams p) {
    using T = typename AccT<MODE>::T;
    constexpr int RPW = 32 / LPR;
    constexpr int SB = LPR * BPL;
    const int lane = threadIdx.x & 31, lg = lane % LPR, grp = lane / LPR;
    const int warp = blockIdx.x * Q8_WARPS + (threadIdx.x >> 5);
    const int W = gridDim.x * Q8_WARPS;
    const int S = p.S;
    const int slice = warp % S;
    const int wstride = (W - slice + S - 1) / S;
    int bidx[BPL];
    bool bval[BPL];
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        bidx[j] = slice * SB + lg + j * LPR;
        bval[j] = bidx[j] < p.nb;
    }
    griddep_wait();
    const int ng = n_groups(p);
    const int items = ng * p.nrs;
    float xf[MODE == 0 ? BPL * 32 : 1];
    uint32_t xw[MODE == 1 ? BPL : 1][8];
    float xsc[BPL];
    int64_t loaded = -1;
    for (int it = warp / S; it < items; it += wstride) {
        const int a = it / p.nrs, rs = it % p.nrs;
        const Group g = group_of(p, a);
        // an expert id outside [0, E) reads no weights and counts as an expert of zero weights
        const bool ev = g.expert >= 0 && g.expert < p.E;
        const int i = rs * RPW + grp;
        const bool rv = i < p.out_rows;
        const int64_t wrow = (int64_t)(ev ? g.expert : 0) * p.out_rows + i;
        uint32_t wg[BPL][8], wu[BPL][8];
        float sg[BPL], su[BPL];
        load_w<MODE, BPL>(p.q0, p.s0, wrow, rv && ev, p.k, p.nb, bidx, bval, wg, sg);
        load_w<MODE, BPL>(p.q1, p.s1, wrow, rv && ev, p.k, p.nb, bidx, bval, wu, su);
        for (int ci = 0; ci < g.nc; ++ci) {
            const int c = choice_of(p, g, ci);
            const int64_t xrow = c / p.K;  // the token row of choice c
            if (xrow != loaded) {
                load_x<MODE, BPL>(p.x, p.xq, p.xs, xrow, p.k, p.nb, bidx, bval, xf, xw, xsc);
                loaded = xrow;
            }
            T gv = group_sum<LPR>(dot<MODE, BPL>(wg, sg, xf, xw, xsc));
            T uv = group_sum<LPR>(dot<MODE, BPL>(wu, su, xf, xw, xsc));
            bool done = true;
            if (S > 1) {
                T* part = reinterpret_cast<T*>(p.partial);  // [R*K][S][2][out_rows]
                if (lg == 0 && rv) {
                    part[(((int64_t)c * S + slice) * 2 + 0) * p.out_rows + i] = gv;
                    part[(((int64_t)c * S + slice) * 2 + 1) * p.out_rows + i] = uv;
                }
                int* cnt = p.cnt_slice + (int64_t)c * p.nrs + rs;
                done = warp_arrive_last(cnt, S);
                if (done) {
                    gv = 0;
                    uv = 0;
                    if (lg == 0 && rv)
                        for (int sl = 0; sl < S; ++sl) {
                            gv += __ldcg(part + (((int64_t)c * S + sl) * 2 + 0) * p.out_rows + i);
                            uv += __ldcg(part + (((int64_t)c * S + sl) * 2 + 1) * p.out_rows + i);
                        }
                    if (lane == 0) *cnt = 0;
                }
            }
            if (done) {
                if (lg == 0 && rv) p.h[(int64_t)c * p.out_rows + i] = silu_f32((float)gv) * (float)uv;
                if (p.hq) {
                    const int i0 = rs * RPW;
                    const int rows = min(RPW, p.out_rows - i0);
                    quant_arrive<RPW>(p, c, i0, rows);
                }
            }
        }
    }
    griddep_launch();
}

// Down-and-combine: item (group a, row-set rs over the d outputs) on slice `slice` of dff; the last of the K*S
// arrivals for (token row r, rs) combines y[r] = residual + sum_j g_j * (sum over slices), j and slices in order.
template <int MODE, int LPR, int BPL>
__global__ void __launch_bounds__(Q8_THREADS, 2) down_kernel(const ExpertParams p) {
    using T = typename AccT<MODE>::T;
    constexpr int RPW = 32 / LPR;
    constexpr int SB = LPR * BPL;
    const int lane = threadIdx.x & 31, lg = lane % LPR, grp = lane / LPR;
    const int warp = blockIdx.x * Q8_WARPS + (threadIdx.x >> 5);
    const int W = gridDim.x * Q8_WARPS;
    const int S = p.S;
    const int slice = warp % S;
    const int wstride = (W - slice + S - 1) / S;
    int bidx[BPL];
    bool bval[BPL];
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        bidx[j] = slice * SB + lg + j * LPR;
        bval[j] = bidx[j] < p.nb;
    }
    griddep_wait();
    const int ng = n_groups(p);
    const int items = ng * p.nrs;
    T* part = reinterpret_cast<T*>(p.partial);  // [R*K][S][out_rows]
    float xf[MODE == 0 ? BPL * 32 : 1];
    uint32_t xw[MODE == 1 ? BPL : 1][8];
    float xsc[BPL];
    for (int it = warp / S; it < items; it += wstride) {
        const int a = it / p.nrs, rs = it % p.nrs;
        const Group g = group_of(p, a);
        const bool ev = g.expert >= 0 && g.expert < p.E;  // see gate_up_kernel
        const int o = rs * RPW + grp;
        const bool rv = o < p.out_rows;
        uint32_t w[BPL][8];
        float sc[BPL];
        load_w<MODE, BPL>(p.q0, p.s0, (int64_t)(ev ? g.expert : 0) * p.out_rows + o, rv && ev, p.k, p.nb, bidx, bval,
                          w, sc);
        for (int ci = 0; ci < g.nc; ++ci) {
            const int c = choice_of(p, g, ci);
            load_x<MODE, BPL>(p.x, p.xq, p.xs, c, p.k, p.nb, bidx, bval, xf, xw, xsc);
            const T acc = group_sum<LPR>(dot<MODE, BPL>(w, sc, xf, xw, xsc));
            if (lg == 0 && rv) part[((int64_t)c * S + slice) * p.out_rows + o] = acc;
            const int r = c / p.K;
            int* cnt = p.cnt_row + (int64_t)r * p.nrs + rs;
            if (warp_arrive_last(cnt, p.K * S)) {
                if (lg == 0 && rv) {
                    T comb = 0;
                    for (int j = 0; j < p.K; ++j) {
                        const int cj = r * p.K + j;
                        T e = 0;
                        for (int sl = 0; sl < S; ++sl) e += __ldcg(part + ((int64_t)cj * S + sl) * p.out_rows + o);
                        if (p.expert_out) p.expert_out[(int64_t)cj * p.out_rows + o] = (float)e;
                        comb += (T)__ldcg(p.gates + cj) * e;
                    }
                    float v = (float)comb;
                    if (p.residual) v = p.residual[(int64_t)r * p.out_rows + o] + v;
                    p.y[(int64_t)r * p.out_rows + o] = v;
                }
                if (lane == 0) *cnt = 0;
            }
        }
    }
    griddep_launch();
}

struct EPlan {
    int lpr, bpl, S;
};

EPlan eplan(int mode, int nb) {
    const int bpl_max = (mode == 0) ? 1 : 2;
    EPlan best{32, 1, 1};
    double best_util = -1.0;
    for (int lpr : {32, 16, 8}) {
        for (int bpl = 1; bpl <= bpl_max; ++bpl) {
            const int sb = lpr * bpl;
            const int S = (nb + sb - 1) / sb;
            const double util = (double)nb / (double)(S * sb);
            if (util > best_util + 1e-9 || (util > best_util - 1e-9 && S < best.S)) {
                best_util = util;
                best = EPlan{lpr, bpl, S};
            }
        }
    }
    return best;
}

int max_groups(const ExpertCall& c) {
    const int64_t choices = c.R * c.K;
    return (int)(choices < c.E ? choices : c.E);
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
    p.xs = c.xs;
    p.h = c.h;
    p.hq = c.hq;
    p.hs = c.hs;
    p.residual = c.residual;
    p.y = c.y;
    p.expert_out = c.expert_out;
    p.S = pl.S;
    p.nrs = (int)((c.out_rows + (32 / pl.lpr) - 1) / (32 / pl.lpr));
    return p;
}

int grid_for(int64_t items, int S) {
    const int64_t max_warps = (int64_t)device_info().sms * 2 * Q8_WARPS;
    int64_t warps = items * S;
    if (warps > max_warps) warps = max_warps;
    if (warps < 1) warps = 1;
    return (int)((warps + Q8_WARPS - 1) / Q8_WARPS);
}

}  // namespace

cudaError_t launch_topk(const TopkCall& c, cudaStream_t st) {
    TopkParams p = {c.logits, (int)c.R, (int)c.E, c.K, c.ids, c.gates,
                    c.plan.counts, c.plan.offsets, c.plan.lists, c.plan.active};
    const size_t smem = c.plan.counts ? (size_t)(2 * c.E + 32) * sizeof(int) : 0;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch(topk_kernel, dim3(1), dim3(TOPK_THREADS), smem, st, c.pdl, p);
}

void gate_up_scratch(const ExpertCall& c, size_t* bytes, size_t* counters) {
    const EPlan pl = eplan(c.mode, (int)(c.k / 32));
    const int64_t nrs = (c.out_rows + (32 / pl.lpr) - 1) / (32 / pl.lpr);
    const int64_t choices = c.R * c.K;
    *bytes = pl.S > 1 ? (size_t)choices * pl.S * 2 * c.out_rows * (c.mode == 0 ? 8 : 4) : 0;
    *counters = (size_t)(pl.S > 1 ? choices * nrs : 0) + (size_t)(c.hq ? choices * (c.out_rows / 32) : 0);
}

void down_scratch(const ExpertCall& c, size_t* bytes, size_t* counters) {
    const EPlan pl = eplan(c.mode, (int)(c.k / 32));
    const int64_t nrs = (c.out_rows + (32 / pl.lpr) - 1) / (32 / pl.lpr);
    *bytes = (size_t)c.R * c.K * pl.S * c.out_rows * (c.mode == 0 ? 8 : 4);
    *counters = (size_t)(c.R * nrs);
}

#define Q8_EXPERT_DISPATCH(KERNEL, MODE)                                                                   \
    if (pl.lpr == 32 && pl.bpl == 1) return launch(KERNEL<MODE, 32, 1>, grid, blk, 0, st, c.pdl, p);     \
    if (pl.lpr == 16 && pl.bpl == 1) return launch(KERNEL<MODE, 16, 1>, grid, blk, 0, st, c.pdl, p);     \
    if (pl.lpr == 8 && pl.bpl == 1) return launch(KERNEL<MODE, 8, 1>, grid, blk, 0, st, c.pdl, p);       \
    if (MODE == 1 && pl.lpr == 32 && pl.bpl == 2) return launch(KERNEL<1, 32, 2>, grid, blk, 0, st, c.pdl, p); \
    if (MODE == 1 && pl.lpr == 16 && pl.bpl == 2) return launch(KERNEL<1, 16, 2>, grid, blk, 0, st, c.pdl, p); \
    if (MODE == 1 && pl.lpr == 8 && pl.bpl == 2) return launch(KERNEL<1, 8, 2>, grid, blk, 0, st, c.pdl, p);

cudaError_t launch_gate_up(const ExpertCall& c, Carve& ws, cudaStream_t st) {
    const EPlan pl = eplan(c.mode, (int)(c.k / 32));
    ExpertParams p = make_params(c, pl);
    const int64_t choices = c.R * c.K;
    if (pl.S > 1) {
        p.partial = ws.take<char>((size_t)choices * pl.S * 2 * c.out_rows * (c.mode == 0 ? 8 : 4));
        p.cnt_slice = ws.take_counters((size_t)(choices * p.nrs));
    }
    if (c.hq) p.cnt_quant = ws.take_counters((size_t)(choices * (c.out_rows / 32)));
    if (ws.overflow) return cudaErrorMemoryAllocation;
    const int grid = grid_for((int64_t)max_groups(c) * p.nrs, pl.S);
    const dim3 blk(Q8_THREADS);
    if (c.mode == 0) {
        Q8_EXPERT_DISPATCH(gate_up_kernel, 0)
    } else {
        Q8_EXPERT_DISPATCH(gate_up_kernel, 1)
    }
    return cudaErrorInvalidConfiguration;
}

cudaError_t launch_down_combine(const ExpertCall& c, Carve& ws, cudaStream_t st) {
    const EPlan pl = eplan(c.mode, (int)(c.k / 32));
    ExpertParams p = make_params(c, pl);
    p.partial = ws.take<char>((size_t)c.R * c.K * pl.S * c.out_rows * (c.mode == 0 ? 8 : 4));
    p.cnt_row = ws.take_counters((size_t)(c.R * p.nrs));
    if (ws.overflow) return cudaErrorMemoryAllocation;
    const int grid = grid_for((int64_t)max_groups(c) * p.nrs, pl.S);
    const dim3 blk(Q8_THREADS);
    if (c.mode == 0) {
        Q8_EXPERT_DISPATCH(down_kernel, 0)
    } else {
        Q8_EXPERT_DISPATCH(down_kernel, 1)
    }
    return cudaErrorInvalidConfiguration;
}

}  // namespace q8
