// The Q8_0 projection y = W x at batch 1 (and a few rows), both numerics, on sm_103a.
//
// What it computes: qwen_emit docs, Q8Ref (W[o][t] = q[o*k+t] * s[o*nb + t/32]) and Q8MatKind; lane/mod.rs module docs
// (f32 activations with f64 sums, or one int8 word per value); lane_link.rs, Link::prim (Gemv; a projection cut along
// k whose last-arriving part adds the parts: gemm_blk_tail) and lane/arena.rs, scratch (tp partials, tc counters).
//
// How (GB300 design): the projection is bound by the weight bytes, so every byte is read once with a 256-bit load —
// one whole Q8_0 block per lane per load — and its scale with a coalesced 32-bit load beside it.  A row is spread over
// LPR lanes (LPR consecutive blocks per load, contiguous in memory); each lane group takes RT consecutive rows per item
// and issues all RT*BPL block loads of the item before multiplying any of them; the activation blocks a lane
// multiplies stay in its registers for every row it visits.  Items are dealt to warps round-robin over a persistent
// grid sized to the SMs.  Only a matrix too short to fill the GPU is cut along k: each slice's partial goes to scratch
// and the last warp to arrive on the item's counter adds the slices in slice order (deterministic) and resets it.
#include "common.cuh"
#include "kernels.h"
#include "stream.cuh"

namespace q8 {

namespace {

struct GemvParams {
    const int8_t* q[3];
    const float* s[3];
    float* y[3];
    const float* res[3];
    int n[3];
    int it0[4];      // first item of each segment (it0[nseg] = total items)
    int row0[3];     // first row of each segment in the concatenated row space
    int nseg;
    int ntot;        // rows of all segments
    int k, nb;
    const float* x;
    const int8_t* xq;
    const int8_t* xl;  // mode 2: the low words
    const float* xs;
    int R;
    int RG;          // activation row groups: warp w takes rows w % RG, w % RG + RG, ... (RG <= warps)
    int S;           // slices along k
    void* partial;   // [R][S][ntot] (f64 in mode 0, f32 in mode 1)
    int* counters;   // [R][items]
    int32_t* dots;
    int32_t* dots_lo;  // mode 2: the low words' block dots
    L2Prefetch pf;
};

template <int MODE, int LPR, int BPL, int RT, bool DOTS>
__global__ void __launch_bounds__(Q8_THREADS, 1) gemv_kernel(const GemvParams p) {
    using T = typename AccType<MODE>::T;
    constexpr int RPW = 32 / LPR;
    constexpr int ROWS = RPW * RT;  // rows per item
    constexpr int SB = LPR * BPL;   // blocks per slice
    const int lane = threadIdx.x & 31;
    const int lg = lane % LPR;
    const int grp = lane / LPR;
    const int warp = blockIdx.x * Q8_WARPS + (threadIdx.x >> 5);
    const int RG = p.RG;
    const int rg = warp % RG;                     // this warp's activation rows: rg, rg + RG, ...
    const int wq = warp / RG, WQ = (gridDim.x * Q8_WARPS) / RG;
    if (wq >= WQ) return;                         // the last warps when RG does not divide the grid's warps
    const int S = p.S;
    const int slice = wq % S;
    const int wstride = (WQ - slice + S - 1) / S;  // warps of this row group serving this slice
    const int nit = p.it0[p.nseg];

    int bidx[BPL];
    bool bval[BPL];
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
        bidx[j] = slice * SB + lg + j * LPR;
        bval[j] = bidx[j] < p.nb;
    }
    issue_l2_prefetch(p.pf);
    // the weights do not depend on earlier kernels: the warp's first tile is read before waiting for them
    const int first = wq / S;
    WTile<BPL, RT> t;
    if (first < nit) {
        int sg = 0;
        while (sg + 1 < p.nseg && first >= p.it0[sg + 1]) ++sg;
        const int row0 = (first - p.it0[sg]) * ROWS + grp * RT;
        load_tile<BPL, RT>(t, p.q[sg], p.s[sg], row0, min(RT, p.n[sg] - row0), p.k, p.nb, bidx, bval);
    }
    griddep_wait();
    griddep_launch();

    // each weight tile is read once and multiplied by the warp's activation rows
    for (int it = first; it < nit; it += wstride) {
        int sg = 0;
        while (sg + 1 < p.nseg && it >= p.it0[sg + 1]) ++sg;
        const int row0 = (it - p.it0[sg]) * ROWS + grp * RT;
        const int nvalid = min(RT, p.n[sg] - row0);
        if (it != first) load_tile<BPL, RT>(t, p.q[sg], p.s[sg], row0, nvalid, p.k, p.nb, bidx, bval);
        for (int r = rg; r < p.R; r += RG) {
            XTile<MODE, BPL> x;
            load_x<MODE, BPL>(x, p.x + (int64_t)r * p.k, p.xq + (int64_t)r * p.k, p.xl + (int64_t)r * p.k,
                              p.xs + (int64_t)r * p.nb, bidx, bval);
            T acc[RT];
#pragma unroll
            for (int i = 0; i < RT; ++i) {
                if (DOTS) {
#pragma unroll
                    for (int j = 0; j < BPL; ++j)
                        if (i < nvalid && bval[j]) {
                            const int64_t at = ((int64_t)r * p.ntot + row0 + i) * p.nb + bidx[j];
                            p.dots[at] = block_dot_i8(t.w[i][j], x.w[j]);
                            if (MODE == 2) p.dots_lo[at] = block_dot_i8(t.w[i][j], x.l[MODE == 2 ? j : 0]);
                        }
                }
                acc[i] = group_sum<LPR>(tile_row_dot<MODE, BPL, RT>(t, i, x));
            }
            if (S == 1) {
                if (lg == 0)
#pragma unroll
                    for (int i = 0; i < RT; ++i)
                        if (i < nvalid) {
                            float v = (float)acc[i];
                            if (p.res[sg]) v = p.res[sg][(int64_t)r * p.n[sg] + row0 + i] + v;
                            p.y[sg][(int64_t)r * p.n[sg] + row0 + i] = v;
                        }
            } else {
                T* part = reinterpret_cast<T*>(p.partial);
                const int grow = p.row0[sg] + row0;
                if (lg == 0)
#pragma unroll
                    for (int i = 0; i < RT; ++i)
                        if (i < nvalid) part[((int64_t)r * S + slice) * p.ntot + grow + i] = acc[i];
                int* cnt = p.counters + (int64_t)r * nit + it;
                if (warp_arrive_last(cnt, S)) {
                    if (lg == 0)
                        for (int i = 0; i < nvalid; ++i) {
                            T sum = 0;
                            for (int sl = 0; sl < S; ++sl)
                                sum += __ldcg(part + ((int64_t)r * S + sl) * p.ntot + grow + i);
                            float v = (float)sum;
                            if (p.res[sg]) v = p.res[sg][(int64_t)r * p.n[sg] + row0 + i] + v;
                            p.y[sg][(int64_t)r * p.n[sg] + row0 + i] = v;
                        }
                    if (lane == 0) *cnt = 0;
                }
            }
        }
    }
}

// ---- the TMA-fed projection (one activation row) -------------------------------------------------------------------
// A CTA owns tiles t = blockIdx.x + i*gridDim.x of TR consecutive rows (never across segments).  Warp 8 lane 0 copies
// each tile's quant rows and scale rows into a ring of NS shared-memory stages with cp.async.bulk; the first NS tiles
// are issued before waiting for earlier kernels, since weights never depend on them.  Warps 0..7 take rows w, w+8, ...
// of a stage: lane l reads the 16 bytes at 16l + 512j of the row (conflict-free), lanes 2m and 2m+1 hold the two halves
// of block m + 16j and add their partial dots with one shuffle before the block is scaled.
constexpr int TMA_CONSUMERS = 8;
constexpr int TMA_THREADS = (TMA_CONSUMERS + 1) * 32;
constexpr int TMA_MAX_TR = 16;
constexpr int TMA_SMEM = 100 * 1024;      // ring of a projection that shares its SMs with the kernel before it
constexpr int TMA_SMEM_BIG = 200 * 1024;  // ring of a matrix of more than 64 MB (the LM head): twice the bytes in flight
constexpr int TMA_MAX_STAGES = 16;
constexpr int TMA_HDR = 2 * TMA_MAX_STAGES * 8;  // the full and empty barriers


// Optional RMSNorm prologue of the TMA projection: x = RMSNorm(a) * w formed by every CTA from the f32 row a (or the
// row a_row of the table a, an embedding gather), kept in shared memory.  CTA 0 writes the gathered row to sum_out.
struct NormIn {
    const float* a;
    const int32_t* a_row;
    int64_t a_rows;
    const float* w;
    float eps;
    float* sum_out;
    int* err;
};

struct TmaParams {
    NormIn ni;
    GemvParams g;
    int tr;        // rows per tile
    int tiles;     // total tiles over all segments
    int t0[4];     // first tile of each segment
    int ns;        // stages
    int stage;     // bytes per stage (quants then scales, 16-byte aligned)
    int* err;
};

template <int MODE, int KCH>
__global__ void __launch_bounds__(TMA_THREADS, 1) gemv_tma_kernel(const TmaParams tp) {
    using T = typename AccType<MODE>::T;
    extern __shared__ __align__(128) unsigned char smem[];
    const GemvParams& p = tp.g;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + TMA_MAX_STAGES;
    unsigned char* ring = smem + TMA_HDR;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int k = p.k, nb = p.nb;
    const int nmine = tp.tiles > (int)blockIdx.x ? (tp.tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < tp.ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], TMA_CONSUMERS);
        }
        fence_barrier_init();
    }
    __syncthreads();
    issue_l2_prefetch(p.pf);

    auto tile_of = [&](int i, int& sg, int& row0, int& rows) {
        const int t = blockIdx.x + i * gridDim.x;
        sg = 0;
        while (sg + 1 < p.nseg && t >= tp.t0[sg + 1]) ++sg;
        row0 = (t - tp.t0[sg]) * tp.tr;
        rows = min(tp.tr, p.n[sg] - row0);
    };

    const NormIn& ni = tp.ni;
    const bool norm = ni.a != nullptr;  // grid-uniform
    constexpr int NP = 2 * KCH;         // 256-value rounds of the row: k <= 512 * KCH
    float nw[NP];
    if (wid == TMA_CONSUMERS) {
        // producer: weights only, so it never waits for earlier kernels; with a norm prologue it first lets the
        // consumers issue their norm-weight loads, so those do not queue behind the bulk copies
        if (norm) asm volatile("bar.sync 2, %0;" ::"n"(TMA_THREADS));
        if (lane == 0) {
            for (int i = 0; i < nmine; ++i) {
                const int s = i % tp.ns;
                if (i >= tp.ns && !mbar_wait(&empty[s], ((i / tp.ns) - 1) & 1, tp.err)) break;
                int sg, row0, rows;
                tile_of(i, sg, row0, rows);
                unsigned char* st = ring + (size_t)s * tp.stage;
                const unsigned qb = (unsigned)rows * (unsigned)k, sb = (unsigned)rows * (unsigned)nb * 4u;
                mbar_arrive_expect_tx(&full[s], qb + sb);
                bulk_g2s(st, p.q[sg] + (int64_t)row0 * k, qb, &full[s]);
                bulk_g2s(st + (size_t)tp.tr * k, p.s[sg] + (int64_t)row0 * nb, sb, &full[s]);
            }
        }
        return;
    }

    if (norm) {
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            const int i = threadIdx.x + TMA_CONSUMERS * 32 * j;
            nw[j] = i < k ? ld_f32_early(ni.w + i) : 0.f;
        }
        asm volatile("bar.arrive 2, %0;" ::"n"(TMA_THREADS));
    }
    griddep_wait();
    griddep_launch();
    const float* xfp = p.x;
    const int8_t* xqp = p.xq;
    const int8_t* xlp = p.xl;
    const float* xsp = p.xs;
    if (norm) {
        // RMSNorm prologue, the same order in every CTA: squares summed as f32 pairs, each y rounded once
        float* xbuf = reinterpret_cast<float*>(ring + (size_t)tp.ns * tp.stage);  // k floats (or k words), then scales
        float* xsbuf = xbuf + k;
        F2* nred = reinterpret_cast<F2*>(xsbuf + k / 32);
        const float* a = ni.a;
        if (ni.a_row) {
            const int32_t idx = *ni.a_row;
            const bool bad = idx < 0 || idx >= ni.a_rows;  // an out-of-range token: flagged, row 0 read instead
            a = ni.a + (int64_t)(bad ? 0 : idx) * k;
            if (bad && blockIdx.x == 0 && threadIdx.x == 0 && ni.err) atomicOr(ni.err, 1);
        }
        float av[NP];
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            const int i = threadIdx.x + TMA_CONSUMERS * 32 * j;
            av[j] = i < k ? __ldcg(a + i) : 0.f;
        }
        F2 ss = f2_two_prod(av[0], av[0]);
#pragma unroll
        for (int j = 1; j < NP; ++j) ss = f2_add(ss, f2_two_prod(av[j], av[j]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            ss = f2_add(ss, F2{__shfl_xor_sync(0xffffffffu, ss.hi, o), __shfl_xor_sync(0xffffffffu, ss.lo, o)});
        if (lane == 0) nred[wid] = ss;
        asm volatile("bar.sync 1, %0;" ::"n"(TMA_CONSUMERS * 32));
        if (threadIdx.x == 0) {
            F2 tot = nred[0];
            for (int w = 1; w < TMA_CONSUMERS; ++w) tot = f2_add(tot, nred[w]);
            const float df = (float)k;
            const float qh = tot.hi / df;
            const float ql = (fmaf(-qh, df, tot.hi) + tot.lo) / df;
            nred[TMA_CONSUMERS] = f2_rsqrt(f2_add(f2_quick(qh, ql), F2{ni.eps, 0.f}));
        }
        asm volatile("bar.sync 1, %0;" ::"n"(TMA_CONSUMERS * 32));
        const F2 inv = nred[TMA_CONSUMERS];
        float y[NP];
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            const int i = threadIdx.x + TMA_CONSUMERS * 32 * j;
            y[j] = f2_mul3_round(av[j], nw[j], inv);
            if (i < k && ni.sum_out && blockIdx.x == 0) ni.sum_out[i] = av[j];
        }
        if (MODE == 0) {
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                const int i = threadIdx.x + TMA_CONSUMERS * 32 * j;
                if (i < k) xbuf[i] = y[j];
            }
        } else if (MODE == 1) {
            int8_t qv[NP];
            float dsc[NP];
            quantize_lanes<NP>(y, qv, dsc);  // round j: warp w holds block w + 8 j
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                const int i = threadIdx.x + TMA_CONSUMERS * 32 * j;
                if (i < k) {
                    reinterpret_cast<int8_t*>(xbuf)[i] = qv[j];
                    if (lane == 0) xsbuf[i / 32] = dsc[j];
                }
            }
        } else {
            int8_t qv[NP], lv[NP];
            float dsc[NP];
            quantize2_lanes<NP>(y, qv, lv, dsc);  // the high words, then the low words k bytes on
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                const int i = threadIdx.x + TMA_CONSUMERS * 32 * j;
                if (i < k) {
                    reinterpret_cast<int8_t*>(xbuf)[i] = qv[j];
                    reinterpret_cast<int8_t*>(xbuf)[k + i] = lv[j];
                    if (lane == 0) xsbuf[i / 32] = dsc[j];
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(TMA_CONSUMERS * 32));
        xfp = xbuf;
        xqp = reinterpret_cast<const int8_t*>(xbuf);
        xlp = reinterpret_cast<const int8_t*>(xbuf) + k;
        xsp = xsbuf;
    }
    // this lane's activation values: columns 16*lane + 512*j
    uint32_t xw[MODE >= 1 ? KCH : 1][4];
    uint32_t xwl[MODE == 2 ? KCH : 1][4];
    float xsc[KCH];
    float xf[MODE == 0 ? KCH : 1][MODE == 0 ? 16 : 1];
#pragma unroll
    for (int j = 0; j < KCH; ++j) {
        const int col = 16 * lane + 512 * j;
        const bool ok = col < k;
        if (MODE >= 1) {
            const uint4 v = ok ? *reinterpret_cast<const uint4*>(xqp + col) : make_uint4(0, 0, 0, 0);
            xw[j][0] = v.x; xw[j][1] = v.y; xw[j][2] = v.z; xw[j][3] = v.w;
            if (MODE == 2) {
                const uint4 u = ok ? *reinterpret_cast<const uint4*>(xlp + col) : make_uint4(0, 0, 0, 0);
                const int jj = MODE == 2 ? j : 0;
                xwl[jj][0] = u.x; xwl[jj][1] = u.y; xwl[jj][2] = u.z; xwl[jj][3] = u.w;
            }
            xsc[j] = ok ? xsp[col / 32] : 0.f;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 v = ok ? *reinterpret_cast<const float4*>(xfp + col + 4 * e) : make_float4(0.f, 0.f, 0.f, 0.f);
                xf[j][4 * e] = v.x; xf[j][4 * e + 1] = v.y; xf[j][4 * e + 2] = v.z; xf[j][4 * e + 3] = v.w;
            }
            xsc[j] = 0.f;
        }
    }
    bool ok_all = true;
    for (int i = 0; i < nmine; ++i) {
        const int s = i % tp.ns;
        if (!mbar_wait(&full[s], (i / tp.ns) & 1, tp.err)) {
            ok_all = false;
            break;
        }
        int sg, row0, rows;
        tile_of(i, sg, row0, rows);
        const int8_t* sq = reinterpret_cast<const int8_t*>(ring + (size_t)s * tp.stage);
        const float* ss = reinterpret_cast<const float*>(ring + (size_t)s * tp.stage + (size_t)tp.tr * k);
        for (int r = wid; r < rows; r += TMA_CONSUMERS) {
            T acc = 0;
#pragma unroll
            for (int j = 0; j < KCH; ++j) {
                const int col = 16 * lane + 512 * j;
                const bool ok = col < k;
                const uint4 w = ok ? *reinterpret_cast<const uint4*>(sq + (size_t)r * k + col) : make_uint4(0, 0, 0, 0);
                const float sc = ok ? ss[(size_t)r * nb + col / 32] : 0.f;
                if (MODE == 1) {
                    int d = __dp4a((int)w.x, (int)xw[j][0], 0);
                    d = __dp4a((int)w.y, (int)xw[j][1], d);
                    d = __dp4a((int)w.z, (int)xw[j][2], d);
                    d = __dp4a((int)w.w, (int)xw[j][3], d);
                    d += __shfl_xor_sync(0xffffffffu, d, 1);  // the block's exact dot: both halves
                    if (!(lane & 1)) acc = fmaf(sc * xsc[j], (float)d, (float)acc);
                } else if (MODE == 2) {
                    const int jj = MODE == 2 ? j : 0;
                    int d = __dp4a((int)w.x, (int)xw[j][0], 0);
                    d = __dp4a((int)w.y, (int)xw[j][1], d);
                    d = __dp4a((int)w.z, (int)xw[j][2], d);
                    d = __dp4a((int)w.w, (int)xw[j][3], d);
                    int e = __dp4a((int)w.x, (int)xwl[jj][0], 0);
                    e = __dp4a((int)w.y, (int)xwl[jj][1], e);
                    e = __dp4a((int)w.z, (int)xwl[jj][2], e);
                    e = __dp4a((int)w.w, (int)xwl[jj][3], e);
                    d = d * 128 + e;
                    d += __shfl_xor_sync(0xffffffffu, d, 1);  // the block's exact two-word dot: both halves
                    if (!(lane & 1)) acc = fmaf(sc * xsc[j] * 0.0078125f, (float)d, (float)acc);
                } else {
                    const uint32_t wv[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u,
                                            w.w ^ 0x80808080u};
                    float p0 = 0.f, p1 = 0.f;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        p0 = fmaf(i8_to_f32<0>(wv[e]), xf[j][4 * e + 0], p0);
                        p1 = fmaf(i8_to_f32<1>(wv[e]), xf[j][4 * e + 1], p1);
                        p0 = fmaf(i8_to_f32<2>(wv[e]), xf[j][4 * e + 2], p0);
                        p1 = fmaf(i8_to_f32<3>(wv[e]), xf[j][4 * e + 3], p1);
                    }
                    float ps = p0 + p1;
                    ps += __shfl_xor_sync(0xffffffffu, ps, 1);  // the block's f32 partial: both halves
                    if (!(lane & 1)) acc = fma((double)sc, (double)ps, (double)acc);
                }
            }
            acc = group_sum<32>(acc);
            if (lane == 0) {
                float v = (float)acc;
                const int row = row0 + r;
                if (p.res[sg]) v = p.res[sg][row] + v;
                p.y[sg][row] = v;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!ok_all)  // a wait gave up: let this CTA's copies in flight land before it exits (again bounded)
        for (int i = 0; i < nmine && i < tp.ns; ++i) mbar_wait(&full[i], 0, nullptr);
}

bool tma_eligible(const GemvCall& c) {
    if (c.R != 1 || c.dots || c.k % 128 != 0 || c.k > 4096) return false;
    if (c.norm_a && c.k % (TMA_CONSUMERS * 32)) return false;
    for (int i = 0; i < c.nseg; ++i)
        if ((uintptr_t)c.seg[i].s % 16 != 0 || (uintptr_t)c.seg[i].q % 16 != 0) return false;
    return true;
}

struct Plan {
    int lpr, bpl, rt, S;
    int RG = 1;  // activation row groups
    int rpw() const { return 32 / lpr; }
    int rows() const { return rpw() * rt; }
};

int items_of(const GemvCall& c, const Plan& pl) {
    int total = 0;
    for (int i = 0; i < c.nseg; ++i) total += (int)((c.seg[i].n + pl.rows() - 1) / pl.rows());
    return total;
}

Plan plan_for(const GemvCall& c) {
    const int nb = (int)(c.k / 32);
    const int bpl_max = (c.mode == 0) ? 3 : 4;  // the int8 modes hold more blocks a lane
    // lanes per row and blocks per lane: the fewest slices, then every lane busy
    Plan best{32, 1, 1, 1 << 30};
    double best_util = -1.0;
    for (int lpr : {32, 16, 8}) {
        for (int bpl = 1; bpl <= bpl_max; ++bpl) {
            const int sb = lpr * bpl;
            const int S = (nb + sb - 1) / sb;
            const double util = (double)nb / (double)(S * sb);
            if (S < best.S || (S == best.S && util > best_util + 1e-9)) {
                best_util = util;
                best = Plan{lpr, bpl, 1, S};
            }
        }
    }
    // rows per item: about eight (int8) or four (f32) 32-byte loads in flight per lane
    const int target = (c.mode == 0) ? 4 : 8;
    const int rt = target / best.bpl;
    best.rt = rt >= 4 ? 4 : (rt >= 2 ? 2 : 1);
    // several activation rows: warps split them (each weight tile is then read once per row group)
    const int sms = device_info().sms;
    best.RG = (int)std::min<int64_t>(c.R, 64);
    int64_t wbytes = 0;
    for (int i = 0; i < c.nseg; ++i) wbytes += c.seg[i].n * c.k;
    while (best.RG > 1 && wbytes * best.RG > (int64_t)256 << 20) best.RG /= 2;  // re-reads stay mostly in L2
    // a matrix too short to fill the GPU: fewer rows per item, then more slices
    while (best.rt > 1 && items_of(c, best) * best.S * best.RG < 4 * sms) best.rt /= 2;
    while (best.bpl > 1 && items_of(c, best) * best.S * best.RG < 2 * sms) {
        best.bpl = (best.bpl + 1) / 2;
        best.S = (nb + best.lpr * best.bpl - 1) / (best.lpr * best.bpl);
    }
    return best;
}

template <int MODE, int LPR, int BPL, int RT, bool DOTS>
cudaError_t run(const GemvParams& p, int64_t warps, cudaStream_t st, int pdl) {
    auto kern = gemv_kernel<MODE, LPR, BPL, RT, DOTS>;
    const int grid = persistent_grid(kern, 0, warps);
    GemvParams q = p;
    if (q.RG > grid * Q8_WARPS) q.RG = grid * Q8_WARPS;
    return launch(kern, dim3(grid), dim3(Q8_THREADS), 0, st, pdl, q);
}

template <int MODE, bool DOTS, int LPR>
cudaError_t dispatch_lpr(const Plan& pl, const GemvParams& p, int64_t grid, cudaStream_t st, int pdl) {
    if (pl.bpl == 1 && pl.rt == 1) return run<MODE, LPR, 1, 1, DOTS>(p, grid, st, pdl);
    if (pl.bpl == 1 && pl.rt == 2) return run<MODE, LPR, 1, 2, DOTS>(p, grid, st, pdl);
    if (pl.bpl == 1 && pl.rt == 4) return run<MODE, LPR, 1, 4, DOTS>(p, grid, st, pdl);
    if (pl.bpl == 2 && pl.rt == 1) return run<MODE, LPR, 2, 1, DOTS>(p, grid, st, pdl);
    if (pl.bpl == 2 && pl.rt == 2) return run<MODE, LPR, 2, 2, DOTS>(p, grid, st, pdl);
    if (pl.bpl == 2 && pl.rt == 4) return run<MODE, LPR, 2, 4, DOTS>(p, grid, st, pdl);
    if (pl.bpl == 3 && pl.rt == 1) return run<MODE, LPR, 3, 1, DOTS>(p, grid, st, pdl);
    if (pl.bpl == 3 && pl.rt == 2) return run<MODE, LPR, 3, 2, DOTS>(p, grid, st, pdl);
    if (MODE >= 1 && pl.bpl == 4 && pl.rt == 1) return run<MODE, LPR, 4, 1, DOTS>(p, grid, st, pdl);
    if (MODE >= 1 && pl.bpl == 4 && pl.rt == 2) return run<MODE, LPR, 4, 2, DOTS>(p, grid, st, pdl);
    return cudaErrorInvalidConfiguration;
}

template <int MODE, bool DOTS>
cudaError_t dispatch(const Plan& pl, const GemvParams& p, int64_t grid, cudaStream_t st, int pdl) {
    if (pl.lpr == 32) return dispatch_lpr<MODE, DOTS, 32>(pl, p, grid, st, pdl);
    if (pl.lpr == 16) return dispatch_lpr<MODE, DOTS, 16>(pl, p, grid, st, pdl);
    return dispatch_lpr<MODE, DOTS, 8>(pl, p, grid, st, pdl);
}

}  // namespace

void gemv_scratch(const GemvCall& c, size_t* bytes, size_t* counters) {
    if (tma_eligible(c)) {  // whole rows through the TMA ring: no scratch
        *bytes = 0;
        *counters = 0;
        return;
    }
    const Plan pl = plan_for(c);
    int64_t ntot = 0;
    for (int i = 0; i < c.nseg; ++i) ntot += c.seg[i].n;
    if (pl.S > 1) {
        *bytes = (size_t)c.R * pl.S * ntot * (c.mode == 0 ? 8 : 4);
        *counters = (size_t)c.R * items_of(c, pl);
    } else {
        *bytes = 0;
        *counters = 0;
    }
}

namespace {

template <int MODE, int KCH>
cudaError_t run_tma(const TmaParams& tp, int grid, size_t smem, cudaStream_t st, int pdl) {
    auto kern = gemv_tma_kernel<MODE, KCH>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch(kern, dim3(grid), dim3(TMA_THREADS), smem, st, pdl, tp);
}

cudaError_t launch_gemv_tma(const GemvCall& c, int* err, cudaStream_t st) {
    TmaParams tp = {};
    tp.ni = NormIn{c.norm_a, c.norm_a_row, c.norm_a_rows, c.norm_w, c.eps, c.norm_sum_out, c.err};
    GemvParams& p = tp.g;
    p.nseg = c.nseg;
    p.k = (int)c.k;
    p.nb = (int)(c.k / 32);
    p.x = c.x;
    p.xq = c.xq;
    p.xl = c.xl;
    p.xs = c.xs;
    p.R = 1;
    p.S = 1;
    p.pf = c.pf;
    int64_t rows_total = 0;
    for (int i = 0; i < c.nseg; ++i) rows_total += c.seg[i].n;
    // rows per tile: about 16 KB of quants per stage; smaller tiles when there are few
    int tr = (int)(16384 / c.k);
    if (tr < 4) tr = 4;
    if (tr > TMA_MAX_TR) tr = TMA_MAX_TR;
    const int sms = device_info().sms;
    while (tr > 2 && rows_total / tr < 2 * sms) tr /= 2;
    int tiles = 0;
    for (int i = 0; i < c.nseg; ++i) {
        p.q[i] = c.seg[i].q;
        p.s[i] = c.seg[i].s;
        p.y[i] = c.seg[i].y;
        p.res[i] = c.seg[i].residual;
        p.n[i] = (int)c.seg[i].n;
        tp.t0[i] = tiles;
        tiles += (int)((c.seg[i].n + tr - 1) / tr);
    }
    tp.t0[c.nseg] = tiles;
    tp.tr = tr;
    tp.tiles = tiles;
    tp.stage = (int)(((size_t)tr * c.k + (size_t)tr * (c.k / 32) * 4 + 127) / 128 * 128);
    const int budget = (double)rows_total * c.k > 64.0 * (1 << 20) ? TMA_SMEM_BIG : TMA_SMEM;
    int ns = (budget - TMA_HDR) / tp.stage;
    if (ns > TMA_MAX_STAGES) ns = TMA_MAX_STAGES;
    if (ns < 2) return cudaErrorInvalidConfiguration;
    tp.ns = ns;
    tp.err = err;
    // the normed activation after the ring: k values (f32) or words (two words: 2k bytes), k/32 scales, the
    // reduction's pairs
    const size_t nbytes = c.norm_a ? (size_t)c.k * 4 + (size_t)(c.k / 32) * 4 + (TMA_CONSUMERS + 1) * sizeof(F2) : 0;
    const size_t smem = TMA_HDR + (size_t)ns * tp.stage + nbytes;
    const int grid = tiles < sms ? tiles : sms;
    const int kch = (int)((c.k + 511) / 512);
    if (c.mode == 2) {
        if (kch <= 1) return run_tma<2, 1>(tp, grid, smem, st, c.pdl);
        if (kch <= 2) return run_tma<2, 2>(tp, grid, smem, st, c.pdl);
        if (kch <= 4) return run_tma<2, 4>(tp, grid, smem, st, c.pdl);
        return run_tma<2, 8>(tp, grid, smem, st, c.pdl);
    }
    if (c.mode == 1) {
        if (kch <= 1) return run_tma<1, 1>(tp, grid, smem, st, c.pdl);
        if (kch <= 2) return run_tma<1, 2>(tp, grid, smem, st, c.pdl);
        if (kch <= 4) return run_tma<1, 4>(tp, grid, smem, st, c.pdl);
        return run_tma<1, 8>(tp, grid, smem, st, c.pdl);
    }
    if (kch <= 1) return run_tma<0, 1>(tp, grid, smem, st, c.pdl);
    if (kch <= 2) return run_tma<0, 2>(tp, grid, smem, st, c.pdl);
    if (kch <= 4) return run_tma<0, 4>(tp, grid, smem, st, c.pdl);
    return run_tma<0, 8>(tp, grid, smem, st, c.pdl);
}

}  // namespace

bool gemv_norm_supported(const GemvCall& c) { return tma_eligible(c); }

// Activation rows from which a dense int8 projection takes the tensor cores (q8_set_tensor_core_rows): -1, the
// default, lets one matrix of at least 2048 x 2048 take them from 32 rows on (measured faster there: 64 rows of a
// 2048 x 4096 projection 32.8 us against 45.2 on the CUDA cores, of 4096 x 2048 30.8 against 51.3; smaller matrices,
// fewer rows and several segments in one call stay faster on the CUDA cores, whose time grows with the rows while the
// tensor-core kernel's has a floor of about 25 us); 0: never; 16..64: every shape from that many rows.
int kDenseMmaMinRows = -1;

static bool dense_on_tensor_cores(const GemvCall& c) {
    if (kDenseMmaMinRows < 0)
        return c.R >= 32 && c.nseg == 1 && c.seg[0].n >= 2048 && c.k >= 2048;
    return kDenseMmaMinRows > 0 && c.R >= kDenseMmaMinRows;
}

cudaError_t launch_gemv(const GemvCall& c, Carve& ws, cudaStream_t st) {
    // 16..64 rows of int8 activations (a prefill chunk, a batch of sequences) can go to the tensor cores, the weight
    // tiles read once for all rows (dense_on_tensor_cores); a workspace without room for the kernel's scratch keeps the
    // CUDA-core form
    const size_t at = (ws.used + 255) & ~size_t(255);
    if (dense_on_tensor_cores(c) && dense_mma_supported(c) && ws.base && at + 4096 + 4 * (size_t)c.R <= ws.size)
        return launch_dense_mma(c, ws, st);
    if (tma_eligible(c))
        return launch_gemv_tma(c, c.err ? c.err : (ws.counters ? ws.counters + ws.n_counters - 1 : nullptr), st);
    if (c.norm_a) return cudaErrorInvalidConfiguration;  // the norm prologue exists in the TMA projection only
    const int nb = (int)(c.k / 32);
    const Plan pl = plan_for(c);
    GemvParams p = {};
    p.nseg = c.nseg;
    int it = 0, row = 0;
    for (int i = 0; i < c.nseg; ++i) {
        p.q[i] = c.seg[i].q;
        p.s[i] = c.seg[i].s;
        p.y[i] = c.seg[i].y;
        p.res[i] = c.seg[i].residual;
        p.n[i] = (int)c.seg[i].n;
        p.it0[i] = it;
        p.row0[i] = row;
        it += (int)((c.seg[i].n + pl.rows() - 1) / pl.rows());
        row += (int)c.seg[i].n;
    }
    p.it0[c.nseg] = it;
    p.ntot = row;
    p.k = (int)c.k;
    p.nb = nb;
    p.x = c.x;
    p.xq = c.xq;
    p.xl = c.xl;
    p.xs = c.xs;
    p.R = (int)c.R;
    p.S = pl.S;
    p.dots = c.dots;
    p.dots_lo = c.dots_lo;
    p.pf = c.pf;
    if (pl.S > 1) {
        size_t bytes = 0, cnt = 0;
        gemv_scratch(c, &bytes, &cnt);
        p.partial = ws.take<char>(bytes);
        p.counters = ws.take_counters(cnt);
        if (ws.overflow) return cudaErrorMemoryAllocation;
    }
    // persistent grid: one warp per (row group, item, slice), at most the CTAs resident at once
    p.RG = pl.RG;
    const int64_t grid = (int64_t)it * pl.S * pl.RG;
    if (c.mode == 0) return dispatch<0, false>(pl, p, grid, st, c.pdl);
    if (c.mode == 2) return c.dots ? dispatch<2, true>(pl, p, grid, st, c.pdl) : dispatch<2, false>(pl, p, grid, st, c.pdl);
    if (c.dots) return dispatch<1, true>(pl, p, grid, st, c.pdl);
    return dispatch<1, false>(pl, p, grid, st, c.pdl);
}

}  // namespace q8
