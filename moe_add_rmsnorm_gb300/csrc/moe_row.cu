// The mixture for one token row, as a decode step runs it: the router projection and its top-k in one cluster
// kernel, and the down-and-combine with every weight row requested before waiting for the kernel that writes the
// hidden rows.
//
// What it computes: forward_shim.rs module docs (a sparse mixture as a top-k router, a gate-up kernel and a
// down-and-combine kernel, its Q8_0 matrices dequantized inside the kernels that read them) and kernel_refusal (Moe
// arms: a softmax router whose kept weights are renormalized, SwiGLU experts, no biases); qwen_emit docs,
// emit_moe_forward (router product, softmax top-K renormalized, weighted combine of the kept experts) and MoeWeights
// (stacked experts: down [E*d, dff] with expert e at row e*d).
//
// How (GB300 design): at batch 1 these launches are latency-bound, so the work is arranged around the dependency wait
// of programmatic dependent launch.  The router rows do not depend on earlier kernels and are loaded before the wait;
// one cluster of 8 CTAs forms all logits, gathers them in CTA 0 through distributed shared memory and ranks them
// there (each expert counts the experts ahead of it), which replaces a second launch and K rounds of warp arg-max.
// Gate-up deals each warp a few consecutive hidden rows and issues all of their weight loads at once.  The
// down-and-combine reads the routing written two launches back, so a warp requests its output row's K*dff/32
// weight blocks (one 256-bit load each) before the wait and only the hidden rows after it.
#include <float.h>

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace q8 {
namespace {

// ==== router projection + top-k ===================================================================================

constexpr int RR_CL = 8;         // CTAs in the cluster
constexpr int RR_THREADS = 256;
constexpr int RR_WARPS = RR_THREADS / 32;
constexpr int RR_MAXE = 1024;    // experts one cluster ranks
constexpr int RR_RW = 2;         // router rows per warp loaded before the wait

constexpr int RR_NPER = 16;      // 256-value rounds of a row the kernel norms itself, at most (d <= 4096)

struct RouteRowParams {
    const int8_t* q;
    const float* s;
    int E, d, nb, K;
    const float* x;
    const int8_t* xq;
    const int8_t* xl;
    const float* xs;
    float* logits;
    int32_t* ids;
    float* gates;
    // when norm_a is set the kernel forms the activation itself: x = RMSNorm(norm_a) * norm_w (int8 form in the int8
    // mode), keeps it in shared memory and writes it to x_out (or xq_out / xs_out) for the launches after it
    const float* norm_a;
    const float* norm_w;
    float eps;
    float* x_out;
    int8_t* xq_out;
    int8_t* xl_out;
    float* xs_out;
    L2Prefetch pf;
};

// Ranking key: a NaN logit ranks below every number (and ties with -inf, broken by index).
__device__ __forceinline__ float rank_key(float v) { return v != v ? -INFINITY : v; }

// CTA c of the cluster owns router rows [c*rpc, (c+1)*rpc); warp w the rows w, w+8, ... of that slice; lane l the
// 32-value blocks l, l+32, ... of a row (the projection's own lane layout, so the logits equal the projection's).
template <int MODE, int BPL>
__global__ void __launch_bounds__(RR_THREADS) route_row_kernel(const RouteRowParams p) {
    __shared__ float own[RR_MAXE / RR_CL];
    __shared__ float all[RR_MAXE];
    __shared__ __align__(16) float key[RR_MAXE];
    __shared__ int cnt0[RR_MAXE];
    __shared__ int cnt1[RR_MAXE];
    __shared__ int kid[32];
    __shared__ float kv[32];
    __shared__ __align__(16) float xbuf[RR_THREADS * RR_NPER];  // the normed activation (f32, or its int8 words)
    __shared__ float xsbuf[RR_THREADS * RR_NPER / 32];
    __shared__ F2 nred[RR_WARPS];
    __shared__ F2 ninv;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int rpc = (p.E + RR_CL - 1) / RR_CL;
    const int r0 = rank * rpc;
    int bidx[BPL];
    bool bval[BPL];
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        bidx[j] = lane + 32 * j;
        bval[j] = bidx[j] < p.nb;
    }
    issue_l2_prefetch(p.pf);
    const bool norm = p.norm_a != nullptr;  // grid-uniform
    constexpr int NP = 4 * BPL;             // 256-value rounds of the row: d <= 1024 * BPL
    float nw[NP];                           // the norm weight, read before the router rows
    if (norm)
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            const int i = threadIdx.x + RR_THREADS * j;
            nw[j] = i < p.d ? ld_f32_early(p.norm_w + i) : 0.f;
        }
    WTile<BPL, 1> t[RR_RW];
#pragma unroll
    for (int u = 0; u < RR_RW; ++u) {
        const int lr = wid + RR_WARPS * u;
        const bool v = lr < rpc && r0 + lr < p.E;
        load_tile<BPL, 1>(t[u], p.q, p.s, v ? r0 + lr : 0, v ? 1 : 0, p.d, p.nb, bidx, bval);
    }
    griddep_wait();  // the activation (or the row it is normed from) comes from the previous launch
    griddep_launch();
    const float* xf = p.x;
    const int8_t* xq = p.xq;
    const int8_t* xl = p.xl;
    const float* xsc = p.xs;
    if (norm) {
        // RMSNorm of the residual row, every CTA of the cluster in the same order (so all hold the same x): the sum
        // of squares and the norm factor in f32 pairs, each y rounded once
        float a[NP];
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            const int i = threadIdx.x + RR_THREADS * j;
            a[j] = i < p.d ? __ldcg(p.norm_a + i) : 0.f;
        }
        F2 ss = f2_two_prod(a[0], a[0]);
#pragma unroll
        for (int j = 1; j < NP; ++j) ss = f2_add(ss, f2_two_prod(a[j], a[j]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            ss = f2_add(ss, F2{__shfl_xor_sync(0xffffffffu, ss.hi, o), __shfl_xor_sync(0xffffffffu, ss.lo, o)});
        if (lane == 0) nred[wid] = ss;
        __syncthreads();
        if (threadIdx.x == 0) {
            F2 tot = nred[0];
            for (int w = 1; w < RR_WARPS; ++w) tot = f2_add(tot, nred[w]);
            const float df = (float)p.d;
            const float qh = tot.hi / df;
            const float ql = (fmaf(-qh, df, tot.hi) + tot.lo) / df;
            ninv = f2_rsqrt(f2_add(f2_quick(qh, ql), F2{p.eps, 0.f}));
        }
        __syncthreads();
        const F2 inv = ninv;
        float y[NP];
#pragma unroll
        for (int j = 0; j < NP; ++j) y[j] = f2_mul3_round(a[j], nw[j], inv);
        if (MODE == 0) {
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                const int i = threadIdx.x + RR_THREADS * j;
                if (i < p.d) {
                    xbuf[i] = y[j];
                    if (j % RR_CL == rank) p.x_out[i] = y[j];  // CTA r writes rounds j = r, r + 8, ...
                }
            }
        } else {
            int8_t qv[NP], lv[NP];
            float dsc[NP];
            if (MODE == 2) quantize2_lanes<NP>(y, qv, lv, dsc);  // round j: warp w holds block w + 8 j
            else quantize_lanes<NP>(y, qv, dsc);
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                const int i = threadIdx.x + RR_THREADS * j;
                if (i < p.d) {
                    reinterpret_cast<int8_t*>(xbuf)[i] = qv[j];
                    if (MODE == 2) reinterpret_cast<int8_t*>(xbuf)[p.d + i] = lv[j];  // the low words d bytes on
                    if (lane == 0) xsbuf[i / 32] = dsc[j];
                    if (j % RR_CL == rank) {  // CTA r writes rounds j = r, r + 8, ...
                        p.xq_out[i] = qv[j];
                        if (MODE == 2) p.xl_out[i] = lv[j];
                        if (lane == 0) p.xs_out[i / 32] = dsc[j];
                    }
                }
            }
        }
        __syncthreads();
        xf = xbuf;
        xq = reinterpret_cast<const int8_t*>(xbuf);
        xl = reinterpret_cast<const int8_t*>(xbuf) + p.d;
        xsc = xsbuf;
    }
    XTile<MODE, BPL> x;
    load_x<MODE, BPL>(x, xf, xq, xl, xsc, bidx, bval);
#pragma unroll
    for (int u = 0; u < RR_RW; ++u) {
        const int lr = wid + RR_WARPS * u;
        const float v = (float)group_sum<32>(tile_row_dot<MODE, BPL, 1>(t[u], 0, x));
        if (lane == 0 && lr < rpc && r0 + lr < p.E) {
            own[lr] = v;
            if (p.logits) p.logits[r0 + lr] = v;
        }
    }
    for (int lr = wid + RR_WARPS * RR_RW; lr < rpc && r0 + lr < p.E; lr += RR_WARPS) {  // past the preloaded rows
        WTile<BPL, 1> w;
        load_tile<BPL, 1>(w, p.q, p.s, r0 + lr, 1, p.d, p.nb, bidx, bval);
        const float v = (float)group_sum<32>(tile_row_dot<MODE, BPL, 1>(w, 0, x));
        if (lane == 0) {
            own[lr] = v;
            if (p.logits) p.logits[r0 + lr] = v;
        }
    }
    cluster.sync();  // every CTA's logits are in its shared memory
    if (rank == 0)
        for (int e = threadIdx.x; e < p.E; e += RR_THREADS) {
            const float v = cluster.map_shared_rank(own, e / rpc)[e % rpc];
            all[e] = v;
            key[e] = rank_key(v);
        }
    cluster.sync();  // CTA 0 has read every slice: the others may leave
    if (rank != 0) return;
    // expert e's place among the kept = the number of experts with a larger key, or an equal key and a lower index;
    // the two halves of the CTA count over the two halves of the experts (keys padded to a multiple of 8 with -inf
    // entries that never count: they sit past every real index)
    const int E8 = (p.E + 7) & ~7;
    for (int e = p.E + threadIdx.x; e < E8; e += RR_THREADS) key[e] = -INFINITY;
    __syncthreads();
    const int half = threadIdx.x / (RR_THREADS / 2), hl = threadIdx.x % (RR_THREADS / 2);
    const int f0 = half ? (E8 / 16) * 8 : 0, f1 = half ? E8 : (E8 / 16) * 8;
    for (int e = hl; e < p.E; e += RR_THREADS / 2) {
        const float ke = key[e];
        int r = 0;
        for (int f = f0; f < f1; f += 8) {
            const float4 a = *reinterpret_cast<const float4*>(key + f);
            const float4 b = *reinterpret_cast<const float4*>(key + f + 4);
            const float kf[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) r += (kf[i] > ke) || (kf[i] == ke && f + i < e);
        }
        if (half) cnt1[e] = r;
        else cnt0[e] = r;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += RR_THREADS) {
        const int r = cnt0[e] + cnt1[e];
        if (r < p.K) {
            kid[r] = e;
            kv[r] = all[e];
        }
    }
    __syncthreads();
    if (wid == 0) {
        // gates: softmax over all experts renormalized over the kept ones = softmax over the kept logits
        const float kept = lane < p.K ? kv[lane] : 0.f;
        const float m = kv[0];
        const float pe = lane < p.K ? expf(kept - m) : 0.f;
        const float z = group_sum<32>(pe);
        if (lane < p.K) {
            p.ids[lane] = kid[lane];
            p.gates[lane] = __fdiv_rn(pe, z);
        }
    }
}

template <int MODE, int BPL>
cudaError_t run_route_row(const RouteRowParams& p, cudaStream_t st, int pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(RR_CL);
    cfg.blockDim = dim3(RR_THREADS);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = RR_CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int na = 1;
    if (pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, route_row_kernel<MODE, BPL>, p);
}

// ==== gate-up ========================================================================================================

constexpr int GR_WPC = 14;  // warps per CTA

struct GateRowParams {
    const int8_t* gq;  // gate and up [E*dff][d]
    const float* gs;
    const int8_t* uq;
    const float* us;
    int E, dff, d, nb, K;
    const int32_t* ids;
    const int8_t* xq;  // int8 modes: the normed activation [d] (mode 2: high words), its low words, its scales
    const int8_t* xl;
    const float* xs;
    float* h;          // [K][dff]
    int8_t* hq;        // optional: h quantized per 32 rows [K][dff] (mode 2: with low words hl) and its scales
    int8_t* hl;        // [K][dff/32] (dff % 32 == 0)
    float* hs;
    int* qcnt;         // [(K*dff + sdff)/32] arrivals per 32-row block (left zero)
    const int8_t* sgq; // a shared expert's gate and up [sdff][d] (sdff > 0): its rows are items K*dff.., its hidden
    const float* sgs;  // rows follow the routed ones in h (and in the int8 forms)
    const int8_t* suq;
    const float* sus;
    int sdff;
    L2Prefetch pf;
};

// Int8 mode, one row: item it = (kept expert it / dff, hidden row it % dff) is that row of the expert's gate and up
// matrices; warp w takes items w*IPW .. w*IPW + IPW - 1 (consecutive rows, so each warp reads contiguous weights) and
// issues all of their loads before it multiplies any, so a whole launch's weights are in flight at once.  The expert
// ids and the activation are read after the wait.
template <int MODE, int BPL, int IPW>
__global__ void __launch_bounds__(GR_WPC * 32, 1) gate_row_kernel(const GateRowParams p) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int warp = blockIdx.x * GR_WPC + wid;
    const int W = gridDim.x * GR_WPC;
    const int nk = p.K * p.dff;  // routed items; the shared expert's rows follow
    const int n = nk + p.sdff;
    int bidx[BPL];
    bool bval[BPL];
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        bidx[j] = lane + 32 * j;
        bval[j] = bidx[j] < p.nb;
    }
    issue_l2_prefetch(p.pf);
    griddep_wait();  // the expert ids (and, when the router launch norms it, the activation) come from the previous launch
    griddep_launch();
    XTile<MODE, BPL> x;
    load_x<MODE, BPL>(x, nullptr, p.xq, p.xl, p.xs, bidx, bval);
    for (int it0 = warp * IPW; it0 < n; it0 += W * IPW) {
        WTile<BPL, 1> tg[IPW], tu[IPW];
        int eid[IPW];  // every item's expert id read before any weight address depends on one
#pragma unroll
        for (int u = 0; u < IPW; ++u) eid[u] = it0 + u < nk ? __ldcg(p.ids + (it0 + u) / p.dff) : -1;
#pragma unroll
        for (int u = 0; u < IPW; ++u) {
            const int it = it0 + u;
            const bool sh = it >= nk && it < n;  // a row of the shared expert
            const int j = it / p.dff, i = it - j * p.dff;
            const int e = eid[u];
            const bool ev = e >= 0 && e < p.E;  // an id outside [0, E) counts as an expert of zero weights
            const int64_t wrow = sh ? (int64_t)(it - nk) : (int64_t)(ev ? e : 0) * p.dff + i;
            load_tile<BPL, 1>(tg[u], sh ? p.sgq : p.gq, sh ? p.sgs : p.gs, wrow, (ev || sh) ? 1 : 0, p.d, p.nb, bidx,
                              bval);
            load_tile<BPL, 1>(tu[u], sh ? p.suq : p.uq, sh ? p.sus : p.us, wrow, (ev || sh) ? 1 : 0, p.d, p.nb, bidx,
                              bval);
        }
#pragma unroll
        for (int u = 0; u < IPW; ++u) {
            const float gv = group_sum<32>(tile_row_dot<MODE, BPL, 1>(tg[u], 0, x));
            const float uv = group_sum<32>(tile_row_dot<MODE, BPL, 1>(tu[u], 0, x));
            if (lane == 0 && it0 + u < n) p.h[it0 + u] = silu_f32(gv) * uv;
        }
        if (p.hq) {
            // the int8 epilogue: every warp arrives on the 32-row blocks its rows belong to (item it is row it % 32 of
            // block it / 32), releasing its rows; the warp that completes a block quantizes it, lane = row
            const int b0 = it0 / 32;
            const int last_it = min(it0 + IPW, n) - 1;
            for (int b = b0; b <= last_it / 32; ++b) {  // at most two blocks
                const int lo = max(it0, b * 32), hi = min(last_it, b * 32 + 31);
                int old = 0;
                __syncwarp();
                if (lane == 0) old = atomic_add_acq_rel_gpu(p.qcnt + b, hi - lo + 1);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old + (hi - lo + 1) == 32) {  // warp-uniform
                    __syncwarp();
                    float dsc;
                    const float hv = __ldcg(p.h + (int64_t)b * 32 + lane);
                    if (MODE == 2) {
                        int8_t lv;
                        p.hq[(int64_t)b * 32 + lane] = quantize2_lane(hv, dsc, lv);
                        p.hl[(int64_t)b * 32 + lane] = lv;
                    } else {
                        p.hq[(int64_t)b * 32 + lane] = quantize_lane(hv, dsc);
                    }
                    if (lane == 0) {
                        p.hs[b] = dsc;
                        p.qcnt[b] = 0;
                    }
                }
            }
        }
    }
}

template <int MODE, int BPL, int IPW>
cudaError_t run_gate_row(const GateRowParams& p, cudaStream_t st, int pdl) {
    const int n = p.K * p.dff + p.sdff;
    int grid = (n + GR_WPC * IPW - 1) / (GR_WPC * IPW);
    const int cap = device_info().sms;
    if (grid > cap) grid = cap;
    return launch(gate_row_kernel<MODE, BPL, IPW>, dim3(grid), dim3(GR_WPC * 32), 0, st, pdl, p);
}

template <int MODE>
cudaError_t dispatch_gate_row(const GateRowParams& p, int bpl, int ipw, cudaStream_t st, int pdl) {
    if (bpl == 1) return ipw == 1 ? run_gate_row<MODE, 1, 1>(p, st, pdl) : ipw == 2 ? run_gate_row<MODE, 1, 2>(p, st, pdl)
                                                                             : run_gate_row<MODE, 1, 3>(p, st, pdl);
    if (bpl == 2) return ipw == 1 ? run_gate_row<MODE, 2, 1>(p, st, pdl) : ipw == 2 ? run_gate_row<MODE, 2, 2>(p, st, pdl)
                                                                             : run_gate_row<MODE, 2, 3>(p, st, pdl);
    return run_gate_row<MODE, 4, 1>(p, st, pdl);
}

// ==== down-and-combine ==============================================================================================

constexpr int DR_MAXW = 14;  // warps per CTA at most (146 registers a thread)
constexpr int DR_MAXP = 8;   // (expert, block) pairs per lane at most: K * dff/32 <= 256
constexpr int DR_QB = 16;    // hidden-row blocks a warp loads at once when it quantizes them

struct DownRowParams {
    const int8_t* q;  // down [E*rows][k]
    const float* s;
    int E, rows, k, nb, K;
    const int32_t* ids;
    const float* gates;
    const float* h;    // the K hidden rows [K][k], f32
    const int8_t* hq;  // int8 modes: their words [K][k] (mode 2: high words, with the low words hl) and scales [K][nb];
    const int8_t* hl;  // when null the CTA quantizes h itself
    const float* hs;
    const float* residual;
    float* y;
    const int8_t* sq;  // a shared expert's down [rows][sk] (sk > 0): its blocks are pairs K*nb.., gate 1, its hidden
    const float* ss;   // row after the routed ones (value K*k + 32 b)
    int sk;
    L2Prefetch pf;
};

// Warp o owns output row o: y[o] = residual[o] + sum_j g_j * (Wd[e_j] row o . h_j).  The row's K*nb (expert, block)
// pairs are dealt to the lanes, pair p = lane + 32 i being block p % nb of kept expert p / nb; the lanes add
// g_j * (block product) for their pairs (f64 in the f32 mode) and the warp sums them.
template <int MODE, int PPL>
__global__ void __launch_bounds__(DR_MAXW * 32, 1) down_row_kernel(const DownRowParams p) {
    extern __shared__ __align__(16) float hsm[];  // f32 mode: the hidden rows
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int o = blockIdx.x * (blockDim.x >> 5) + wid;
    const bool orow = o < p.rows;
    const int PK = p.K * p.nb;     // routed pairs
    const int P = PK + p.sk / 32;  // and the shared expert's blocks
    uint32_t w[PPL][8];
    float sw[PPL], g[PPL];
    int xo[PPL];  // the pair's first value in the hidden rows: j*k + 32*b
    issue_l2_prefetch(p.pf);
    // the residual row was written three launches back, before the launch before this one passed its wait: read
    // first, ahead of the weight rows
    const float res = (p.residual && orow && lane == 0) ? ld_f32_early(p.residual + o) : 0.f;
    // the routing was written two launches back, before the previous kernel passed its own wait
#pragma unroll
    for (int i = 0; i < PPL; ++i) {
        const int pi = lane + 32 * i;
        const bool in = orow && pi < PK;
        const bool sh = orow && pi >= PK && pi < P;  // a block of the shared expert
        const int j = in ? pi / p.nb : 0;
        const int b = in ? pi - j * p.nb : 0;
        const int e = in ? __ldg(p.ids + j) : -1;
        // = j*k + 32*b for a routed pair, K*k + 32*(pi - PK) for a shared block; 0 for a lane past the pairs, whose
        // (zero-weight) block is still read in the f32 mode: it must stay inside the staged rows
        xo[i] = (in || sh) ? 32 * pi : 0;
        g[i] = in ? __ldg(p.gates + j) : sh ? 1.f : 0.f;
        if (sh) {
            const int bs = pi - PK;
            ld_block_stream(p.sq + (int64_t)o * p.sk + 32 * bs, w[i]);
            sw[i] = ld_scale_stream(p.ss + (int64_t)o * (p.sk / 32) + bs);
        } else if (e >= 0 && e < p.E) {  // an id outside [0, E) counts as an expert of zero weights
            const int64_t row = (int64_t)e * p.rows + o;
            ld_block_stream(p.q + row * p.k + 32 * b, w[i]);
            sw[i] = ld_scale_stream(p.s + row * p.nb + b);
        } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) w[i][c] = 0u;
            sw[i] = 0.f;
        }
    }
    griddep_wait();  // the hidden rows come from the previous launch
    griddep_launch();
    const int8_t* hq = p.hq;
    const int8_t* hl = p.hl;
    const float* hs = p.hs;
    if (MODE == 0) {
        for (int i = threadIdx.x; i < P * 8; i += blockDim.x)
            reinterpret_cast<float4*>(hsm)[i] = __ldcg(reinterpret_cast<const float4*>(p.h) + i);
        __syncthreads();
    } else if (!hq) {
        // the CTA quantizes the f32 hidden rows into shared memory: warp w takes blocks w, w + W, ..., up to
        // DR_QB of them with every load in flight before the first is quantized
        int8_t* sq = reinterpret_cast<int8_t*>(hsm);
        int8_t* sl = sq + P * 32;                         // mode 2: the low words after the high words
        float* ss = hsm + P * 8 * (MODE == 2 ? 2 : 1);    // then the scales
        const int W = blockDim.x >> 5;
        for (int b0 = wid; b0 < P; b0 += DR_QB * W) {
            float v[DR_QB];
#pragma unroll
            for (int u = 0; u < DR_QB; ++u) {
                const int b = b0 + u * W;
                v[u] = b < P ? __ldcg(p.h + (int64_t)b * 32 + lane) : 0.f;
            }
            int8_t qv[DR_QB], lv[DR_QB];
            float dsc[DR_QB];
            if (MODE == 2) quantize2_lanes<DR_QB>(v, qv, lv, dsc);  // the blocks' warp reductions interleaved
            else quantize_lanes<DR_QB>(v, qv, dsc);
#pragma unroll
            for (int u = 0; u < DR_QB; ++u) {
                const int b = b0 + u * W;
                if (b < P) {
                    sq[b * 32 + lane] = qv[u];
                    if (MODE == 2) sl[b * 32 + lane] = lv[u];
                    if (lane == 0) ss[b] = dsc[u];
                }
            }
        }
        __syncthreads();
        hq = sq;
        hl = sl;
        hs = ss;
    }
    typename AccType<MODE>::T acc = 0;
#pragma unroll
    for (int i = 0; i < PPL; ++i) {
        const bool in = orow && lane + 32 * i < P;
        if (MODE >= 1) {  // P words and scales: the routed pairs' hidden blocks, then the shared expert's
            uint32_t xw[8], xl[8];
            float xs = 0.f;
            if (in) {  // global (written by the previous launch) or this CTA's shared memory
                load_words32(hq + xo[i], xw);
                if (MODE == 2) load_words32(hl + xo[i], xl);
                xs = hs[xo[i] / 32];
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) xw[c] = xl[c] = 0u;
            }
            if (MODE == 2) {
                const int D = block_dot_i8x2(w[i], xw, xl);
                acc = fmaf(g[i] * (sw[i] * xs * 0.0078125f), (float)D, (float)acc);
            } else {
                const int D = block_dot_i8(w[i], xw);
                acc = fmaf(g[i] * (sw[i] * xs), (float)D, (float)acc);
            }
        } else {
            float xf[32];
            const float4* src = reinterpret_cast<const float4*>(hsm + xo[i]);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 v = src[c];
                xf[4 * c] = v.x;
                xf[4 * c + 1] = v.y;
                xf[4 * c + 2] = v.z;
                xf[4 * c + 3] = v.w;
            }
            const float ps = block_dot_f32(w[i], xf);
            acc = fma((double)g[i] * (double)sw[i], (double)ps, (double)acc);
        }
    }
    acc = group_sum<32>(acc);
    if (lane == 0 && orow) {
        float v = (float)acc;
        if (p.residual) v = res + v;
        p.y[o] = v;
    }
}

template <int MODE, int PPL>
cudaError_t run_down_row(const DownRowParams& p, int wpc, cudaStream_t st, int pdl) {
    auto kern = down_row_kernel<MODE, PPL>;
    const size_t vals = (size_t)p.K * p.k + p.sk;  // the hidden values the kernel reads
    const size_t smem = MODE == 0 ? vals * sizeof(float) : p.hq ? 0 : vals * (MODE == 2 ? 2 : 1) + vals / 32 * 4 + 16;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const int grid = (p.rows + wpc - 1) / wpc;
    return launch(kern, dim3(grid), dim3(wpc * 32), smem, st, pdl, p);
}

template <int MODE>
cudaError_t dispatch_down_row(const DownRowParams& p, int ppl, int wpc, cudaStream_t st, int pdl) {
    switch (ppl) {
        case 1: return run_down_row<MODE, 1>(p, wpc, st, pdl);
        case 2: return run_down_row<MODE, 2>(p, wpc, st, pdl);
        case 3: return run_down_row<MODE, 3>(p, wpc, st, pdl);
        case 4: return run_down_row<MODE, 4>(p, wpc, st, pdl);
        case 5: return run_down_row<MODE, 5>(p, wpc, st, pdl);
        case 6: return run_down_row<MODE, 6>(p, wpc, st, pdl);
        case 7: return run_down_row<MODE, 7>(p, wpc, st, pdl);
        case 8: return run_down_row<MODE, 8>(p, wpc, st, pdl);
    }
    return cudaErrorInvalidConfiguration;
}

int route_bpl(int mode, int64_t d) {
    const int64_t nb = d / 32;
    const int bpl = nb <= 32 ? 1 : nb <= 64 ? 2 : nb <= 128 ? 4 : 0;
    return (mode == 0 && bpl > 2) ? 0 : bpl;
}

}  // namespace

bool route_row_supported(int mode, int64_t E, int64_t d, int K) {
    return E >= 1 && E <= RR_MAXE && K >= 1 && K <= 32 && K <= E && d % 32 == 0 && route_bpl(mode, d) > 0;
}

cudaError_t launch_route_row(const RouteRowCall& c, cudaStream_t st) {
    if (!route_row_supported(c.mode, c.E, c.d, c.K)) return cudaErrorInvalidConfiguration;
    if (c.norm_a && (c.d % RR_THREADS || c.d > RR_THREADS * RR_NPER || !c.norm_w ||
                     (c.mode == 0 ? !c.x_out : (!c.xq_out || !c.xs_out || (c.mode == 2 && !c.xl_out)))))
        return cudaErrorInvalidValue;
    RouteRowParams p = {c.q, c.s, (int)c.E, (int)c.d, (int)(c.d / 32), c.K, c.x, c.xq, c.xl, c.xs, c.logits, c.ids,
                        c.gates, c.norm_a, c.norm_w, c.eps, c.x_out, c.xq_out, c.xl_out, c.xs_out, c.pf};
    const int bpl = route_bpl(c.mode, c.d);
    if (c.mode == 0) {
        if (bpl == 1) return run_route_row<0, 1>(p, st, c.pdl);
        if (bpl == 2) return run_route_row<0, 2>(p, st, c.pdl);
    } else if (c.mode == 1) {
        if (bpl == 1) return run_route_row<1, 1>(p, st, c.pdl);
        if (bpl == 2) return run_route_row<1, 2>(p, st, c.pdl);
        if (bpl == 4) return run_route_row<1, 4>(p, st, c.pdl);
    } else {
        if (bpl == 1) return run_route_row<2, 1>(p, st, c.pdl);
        if (bpl == 2) return run_route_row<2, 2>(p, st, c.pdl);
        if (bpl == 4) return run_route_row<2, 4>(p, st, c.pdl);
    }
    return cudaErrorInvalidConfiguration;
}

bool gate_row_supported(const ExpertCall& c) {
    return c.mode >= 1 && c.R == 1 && !c.plan.active && c.xq && c.xs && (c.mode == 1 || c.xl) && c.k % 32 == 0 &&
           c.k / 32 <= 128 && c.sdff % 32 == 0 && c.K * c.out_rows + c.sdff < (int64_t(1) << 31) &&
           c.K >= 1 && c.out_rows >= 1 && c.E * c.out_rows < (int64_t(1) << 31);
}

cudaError_t launch_gate_row(const ExpertCall& c, Carve& ws, cudaStream_t st) {
    if (!gate_row_supported(c)) return cudaErrorInvalidConfiguration;
    GateRowParams p = {c.q0, c.s0, c.q1, c.s1, (int)c.E, (int)c.out_rows, (int)c.k, (int)(c.k / 32), c.K, c.ids,
                       c.xq, c.xl, c.xs, c.h, nullptr, nullptr, nullptr, nullptr, c.sq0, c.ss0, c.sq1, c.ss1,
                       (int)c.sdff, c.pf};
    if (c.hq_out) {
        if (c.out_rows % 32 || (c.mode == 2 && !c.hl_out)) return cudaErrorInvalidValue;
        p.hq = c.hq_out;
        p.hl = c.hl_out;
        p.hs = c.hs_out;
        p.qcnt = ws.take_counters((size_t)((c.K * c.out_rows + c.sdff) / 32));
        if (ws.overflow) return cudaErrorMemoryAllocation;
    }
    const int nb = (int)(c.k / 32);
    const int bpl = nb <= 32 ? 1 : nb <= 64 ? 2 : 4;
    // items per warp: enough that one pass covers every item on a grid of one CTA per SM, at most 6 blocks per lane
    const int64_t n = (int64_t)c.K * c.out_rows + c.sdff;
    const int64_t slots = (int64_t)device_info().sms * GR_WPC;
    int ipw = (int)((n + slots - 1) / slots);
    const int ipw_max = bpl == 4 ? 1 : 3;
    if (ipw > ipw_max) ipw = ipw_max;
    return c.mode == 2 ? dispatch_gate_row<2>(p, bpl, ipw, st, c.pdl) : dispatch_gate_row<1>(p, bpl, ipw, st, c.pdl);
}

bool down_row_supported(const ExpertCall& c) {
    const bool act = c.mode == 0 ? (c.x != nullptr && (size_t)(c.K * c.k + c.sdff) * 4 <= 96 * 1024)
                                 : ((c.xq != nullptr && (c.mode == 1 || c.xl != nullptr)) || c.x != nullptr);
    return c.R == 1 && !c.plan.active && !c.expert_out && act && c.k % 32 == 0 && c.K >= 1 && c.sdff % 32 == 0 &&
           (int64_t)c.K * (c.k / 32) + c.sdff / 32 <= 32 * DR_MAXP;
}

cudaError_t launch_down_row(const ExpertCall& c, cudaStream_t st) {
    if (!down_row_supported(c)) return cudaErrorInvalidConfiguration;
    DownRowParams p = {c.q0, c.s0, (int)c.E, (int)c.out_rows, (int)c.k, (int)(c.k / 32), c.K, c.ids, c.gates,
                       c.x, c.xq, c.xl, c.xs, c.residual, c.y, c.sq0, c.ss0, (int)c.sdff, c.pf};
    const int ppl = (int)((c.K * (c.k / 32) + c.sdff / 32 + 31) / 32);
    // one output row per warp, the rows spread over every SM
    const int sms = device_info().sms;
    int wpc = (int)((c.out_rows + sms - 1) / sms);
    if (wpc < 4) wpc = 4;
    if (wpc > DR_MAXW) wpc = DR_MAXW;
    if (c.mode == 2) return dispatch_down_row<2>(p, ppl, wpc, st, c.pdl);
    return c.mode == 0 ? dispatch_down_row<0>(p, ppl, wpc, st, c.pdl) : dispatch_down_row<1>(p, ppl, wpc, st, c.pdl);
}

}  // namespace q8
