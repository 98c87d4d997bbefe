// The Q8_0 projection y = W x at batch 1 (and a few rows), both numerics, on sm_103a.
//
// What it computes: qwen_emit docs, Q8Ref (W[o][t] = q[o*k+t] * s[o*nb + t/32]) and Q8MatKind; lane/mod.rs module docs
// (f32 activations with f64 sums, or one int8 word per value); lane_link.rs, Link::prim (Gemv; a projection cut along
// k whose last-arriving part adds the parts: gemm_blk_tail) and lane/arena.rs, scratch (tp partials, tc counters).
//
// How (GB300 design): the projection is bound by the weight bytes, so every byte is read once with a 256-bit load —
// one whole Q8_0 block per lane per load — and its scale with a coalesced 32-bit load beside it.  A row is spread over
// LPR lanes (LPR consecutive blocks per load, contiguous in memory); the activation blocks a lane multiplies stay in
// its registers for every row it visits.  Rows are dealt to warps round-robin over a persistent grid sized to the SMs.
// When a row is wider than LPR*BPL blocks it is cut into slices; each slice's partial goes to scratch and the last warp
// to arrive on the row-set's counter adds the slices in slice order (deterministic) and resets the counter.
#include "common.cuh"
#include "kernels.h"

namespace q8 {

namespace {

struct GemvParams {
    const int8_t* q[3];
    const float* s[3];
    float* y[3];
    const float* res[3];
    int n[3];
    int rs0[4];      // first row-set of each segment (rs0[nseg] = total row-sets)
    int row0[3];     // first row of each segment in the concatenated row space
    int nseg;
    int ntot;        // rows of all segments
    int k, nb;
    const float* x;
    const int8_t* xq;
    const float* xs;
    int R;
    int S;           // slices along k
    void* partial;   // [R][S][ntot] (f64 in mode 0, f32 in mode 1)
    int* counters;   // [R][row-sets]
    int32_t* dots;
};

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

template <int MODE>
struct Acc;
template <>
struct Acc<0> {
    using T = double;
};
template <>
struct Acc<1> {
    using T = float;
};

// MODE: 0 = f32 activations / f64 sums, 1 = int8 activations.  LPR lanes per row, BPL blocks per lane per slice, U
// row-sets in flight per warp.
template <int MODE, int LPR, int BPL, int U, bool DOTS>
__global__ void __launch_bounds__(Q8_THREADS) gemv_kernel(const GemvParams p) {
    using T = typename Acc<MODE>::T;
    constexpr int RPW = 32 / LPR;
    constexpr int SB = LPR * BPL;
    const int lane = threadIdx.x & 31;
    const int lg = lane % LPR;
    const int grp = lane / LPR;
    const int warp = blockIdx.x * Q8_WARPS + (threadIdx.x >> 5);
    const int W = gridDim.x * Q8_WARPS;
    const int S = p.S;
    const int slice = warp % S;
    const int wstride = (W - slice + S - 1) / S;  // warps serving this slice
    const int nrs = p.rs0[p.nseg];

    int bidx[BPL];
    bool bval[BPL];
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        bidx[j] = slice * SB + lg + j * LPR;
        bval[j] = bidx[j] < p.nb;
    }

    // The weights do not depend on earlier kernels: warm L2 with this warp's first rows before waiting.
    {
        const int rs = warp / S;
        if (rs < nrs) {
            int sg = 0;
            while (sg + 1 < p.nseg && rs >= p.rs0[sg + 1]) ++sg;
            const int row = (rs - p.rs0[sg]) * RPW + grp;
            if (row < p.n[sg] && bval[0])
                asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p.q[sg] + (int64_t)row * p.k + bidx[0] * 32));
        }
    }
    griddep_wait();

    for (int r = 0; r < p.R; ++r) {
        // this lane's activation blocks
        float xf[MODE == 0 ? BPL * 32 : 1];
        uint32_t xw[MODE == 1 ? BPL : 1][8];
        float xsc[BPL];
#pragma unroll
        for (int j = 0; j < BPL; ++j) {
            if (MODE == 0) {
                const float4* xp = reinterpret_cast<const float4*>(p.x + (int64_t)r * p.k + bidx[j] * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float4 v = bval[j] ? __ldg(xp + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                    xf[j * 32 + 4 * i + 0] = v.x;
                    xf[j * 32 + 4 * i + 1] = v.y;
                    xf[j * 32 + 4 * i + 2] = v.z;
                    xf[j * 32 + 4 * i + 3] = v.w;
                }
                xsc[j] = 0.f;
            } else {
                if (bval[j]) {
                    ld_block_shared_use(p.xq + (int64_t)r * p.k + bidx[j] * 32, xw[j]);
                    xsc[j] = __ldg(p.xs + (int64_t)r * p.nb + bidx[j]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) xw[j][i] = 0u;
                    xsc[j] = 0.f;
                }
            }
        }

        for (int rs_base = warp / S; rs_base < nrs; rs_base += U * wstride) {
            uint32_t w[U][BPL][8];
            float sc[U][BPL];
            int seg[U], row[U];
            bool rv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int rs = rs_base + u * wstride;
                int sg = 0;
                while (sg + 1 < p.nseg && rs >= p.rs0[sg + 1]) ++sg;
                seg[u] = sg;
                row[u] = (rs - p.rs0[sg]) * RPW + grp;
                rv[u] = rs < nrs && row[u] < p.n[sg];
#pragma unroll
                for (int j = 0; j < BPL; ++j) {
                    if (rv[u] && bval[j]) {
                        ld_block_stream(p.q[sg] + (int64_t)row[u] * p.k + bidx[j] * 32, w[u][j]);
                        sc[u][j] = ld_scale_stream(p.s[sg] + (int64_t)row[u] * p.nb + bidx[j]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) w[u][j][i] = 0u;
                        sc[u][j] = 0.f;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int rs = rs_base + u * wstride;
                if (rs >= nrs) break;  // warp-uniform
                T acc = 0;
#pragma unroll
                for (int j = 0; j < BPL; ++j) {
                    if (MODE == 0) {
                        const float ps = block_dot_f32(w[u][j], &xf[j * 32]);
                        acc = fma((double)sc[u][j], (double)ps, (double)acc);
                    } else {
                        const int D = block_dot_i8(w[u][j], xw[j]);
                        if (DOTS && rv[u] && bval[j])
                            p.dots[((int64_t)r * p.ntot + row[u]) * p.nb + bidx[j]] = D;
                        acc = fmaf(sc[u][j] * xsc[j], (float)D, (float)acc);
                    }
                }
                acc = group_sum<LPR>(acc);
                const int sg = seg[u];
                if (S == 1) {
                    if (lg == 0 && rv[u]) {
                        float v = (float)acc;
                        if (p.res[sg]) v = p.res[sg][(int64_t)r * p.n[sg] + row[u]] + v;
                        p.y[sg][(int64_t)r * p.n[sg] + row[u]] = v;
                    }
                } else {
                    T* part = reinterpret_cast<T*>(p.partial);
                    const int grow = p.row0[sg] + row[u];
                    if (lg == 0 && rv[u]) part[((int64_t)r * S + slice) * p.ntot + grow] = acc;
                    int* cnt = p.counters + (int64_t)r * nrs + rs;
                    if (warp_arrive_last(cnt, S)) {
                        if (lg == 0 && rv[u]) {
                            T sum = 0;
                            for (int sl = 0; sl < S; ++sl) sum += __ldcg(part + ((int64_t)r * S + sl) * p.ntot + grow);
                            float v = (float)sum;
                            if (p.res[sg]) v = p.res[sg][(int64_t)r * p.n[sg] + row[u]] + v;
                            p.y[sg][(int64_t)r * p.n[sg] + row[u]] = v;
                        }
                        if (lane == 0) *cnt = 0;
                    }
                }
            }
        }
    }
    griddep_launch();
}

struct Plan {
    int lpr, bpl, S, U, rpw;
};

Plan plan_for(int mode, int nb) {
    // lanes per row and blocks per lane: use every lane (no idle block slots), then the fewest slices
    const int bpl_max = (mode == 0) ? 1 : 2;
    Plan best{32, 1, 1, 2, 1};
    double best_util = -1.0;
    for (int lpr : {32, 16, 8}) {
        for (int bpl = 1; bpl <= bpl_max; ++bpl) {
            const int sb = lpr * bpl;
            const int S = (nb + sb - 1) / sb;
            const double util = (double)nb / (double)(S * sb);
            if (util > best_util + 1e-9 || (util > best_util - 1e-9 && S < best.S)) {
                best_util = util;
                best = Plan{lpr, bpl, S, 2, 32 / lpr};
            }
        }
    }
    return best;
}

template <int MODE, int LPR, int BPL, int U, bool DOTS>
cudaError_t run(const GemvParams& p, int grid, cudaStream_t st, int pdl) {
    return launch(gemv_kernel<MODE, LPR, BPL, U, DOTS>, dim3(grid), dim3(Q8_THREADS), 0, st, pdl, p);
}

template <int MODE, bool DOTS>
cudaError_t dispatch(const Plan& pl, const GemvParams& p, int grid, cudaStream_t st, int pdl) {
#define Q8_CASE(L, B)                                                            \
    if (pl.lpr == L && pl.bpl == B) return run<MODE, L, B, 2, DOTS>(p, grid, st, pdl);
    Q8_CASE(32, 1)
    Q8_CASE(16, 1)
    Q8_CASE(8, 1)
    if (MODE == 1) {
        Q8_CASE(32, 2)
        Q8_CASE(16, 2)
        Q8_CASE(8, 2)
    }
#undef Q8_CASE
    return cudaErrorInvalidConfiguration;
}

int rowsets(const GemvCall& c, const Plan& pl) {
    int total = 0;
    for (int i = 0; i < c.nseg; ++i) total += (int)((c.seg[i].n + pl.rpw - 1) / pl.rpw);
    return total;
}

}  // namespace

void gemv_scratch(const GemvCall& c, size_t* bytes, size_t* counters) {
    const Plan pl = plan_for(c.mode, (int)(c.k / 32));
    int64_t ntot = 0;
    for (int i = 0; i < c.nseg; ++i) ntot += c.seg[i].n;
    if (pl.S > 1) {
        *bytes = (size_t)c.R * pl.S * ntot * (c.mode == 0 ? 8 : 4);
        *counters = (size_t)c.R * rowsets(c, pl);
    } else {
        *bytes = 0;
        *counters = 0;
    }
}

cudaError_t launch_gemv(const GemvCall& c, Carve& ws, cudaStream_t st) {
    const int nb = (int)(c.k / 32);
    const Plan pl = plan_for(c.mode, nb);
    GemvParams p = {};
    p.nseg = c.nseg;
    int rs = 0, row = 0;
    for (int i = 0; i < c.nseg; ++i) {
        p.q[i] = c.seg[i].q;
        p.s[i] = c.seg[i].s;
        p.y[i] = c.seg[i].y;
        p.res[i] = c.seg[i].residual;
        p.n[i] = (int)c.seg[i].n;
        p.rs0[i] = rs;
        p.row0[i] = row;
        rs += (int)((c.seg[i].n + pl.rpw - 1) / pl.rpw);
        row += (int)c.seg[i].n;
    }
    p.rs0[c.nseg] = rs;
    p.ntot = row;
    p.k = (int)c.k;
    p.nb = nb;
    p.x = c.x;
    p.xq = c.xq;
    p.xs = c.xs;
    p.R = (int)c.R;
    p.S = pl.S;
    p.dots = c.dots;
    if (pl.S > 1) {
        size_t bytes = 0, cnt = 0;
        gemv_scratch(c, &bytes, &cnt);
        p.partial = ws.take<char>(bytes);
        p.counters = ws.take_counters(cnt);
        if (ws.overflow) return cudaErrorMemoryAllocation;
    }
    // persistent grid: enough warps for every (row-set, slice) item, at most 4 CTAs per SM
    const int64_t items = (int64_t)rs * pl.S;
    const int64_t max_warps = (int64_t)device_info().sms * 4 * Q8_WARPS;
    int64_t warps = items < max_warps ? items : max_warps;
    if (warps < 1) warps = 1;
    const int grid = (int)((warps + Q8_WARPS - 1) / Q8_WARPS);
    if (c.mode == 0) return dispatch<0, false>(pl, p, grid, st, c.pdl);
    if (c.dots) return dispatch<1, true>(pl, p, grid, st, c.pdl);
    return dispatch<1, false>(pl, p, grid, st, c.pdl);
}

}  // namespace q8
