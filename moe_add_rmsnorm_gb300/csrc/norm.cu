// Residual add + RMSNorm with the int8 epilogue, and the standalone activation quantizer.
//
// What it computes: forward_shim.rs module docs (a sum and the RMS norm of it as one row kernel writing the sum on; the
// activation a Q8_0 projection reads quantized in its producer's epilogue), ForwardShim::fits (AddNorm) and
// ForwardShim::supports (the residual summed in f32, uncompensated); lane_link.rs, Link::prim (Norm{x, add, w, rows,
// cols, eps}; the standalone Quant launch).
//
// How: one row per thread-block cluster of up to 8 CTAs (the kernel is latency-bound; its pair arithmetic is spread over 8
// SMs).  A warp holds 32 consecutive values per step, so each 32-value quantisation block is one warp's registers and
// its maximum one warp reduction.  The mean of squares and the norm factor are carried to about 44 bits in pairs of
// f32 (FP64 is slow on this part), so y is rounded to f32 once.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace q8 {
namespace {


constexpr int NORM_THREADS = 256;
constexpr int NORM_MAX_D = 8192;

struct NormParams {
    const float* a;
    const int32_t* a_row;
    int64_t a_rows;
    const float* b;
    const float* w;
    int d;
    float eps;
    float* sum;
    float* y;
    int8_t* yq;
    int8_t* yl;  // with yq: the low words of the two-word form
    float* ys;
    int* err;
    L2Prefetch pf;
};

// One row per cluster of CL CTAs (distributed shared memory, sm_90+): CTA c of the cluster owns the contiguous slice
// [c*d/CL, (c+1)*d/CL) of the row, PER values per thread.  Each CTA sums its squares exactly as products into a pair of
// f32 (about 44 significant bits); the CL partial sums are read through distributed shared memory after a cluster
// barrier and added in rank order by every CTA, so every CTA holds the same norm factor (also a pair) and rounds each
// y = s * inv * w once.  The cluster's second barrier is split: a CTA arrives once it has read the others' sums and
// waits only before it exits.
template <int PER, int CL>
__global__ void __launch_bounds__(NORM_THREADS) add_rmsnorm_kernel(const NormParams p) {
    __shared__ F2 red[NORM_THREADS / 32];
    __shared__ F2 part;
    __shared__ F2 inv_s;
    cg::cluster_group cluster = cg::this_cluster();
    const int crank = (int)cluster.block_rank();
    const int r = blockIdx.x / CL;
    const int t = threadIdx.x;
    const int lane = t & 31, wid = t >> 5;
    const int dl = p.d / CL;  // this CTA's slice
    const int base = crank * dl;
    issue_l2_prefetch(p.pf);
    float wv[PER];  // the norm weight does not depend on earlier kernels: read it before waiting for them
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = j * NORM_THREADS + t;
        wv[j] = i < dl ? p.w[base + i] : 0.f;
    }
    griddep_wait();
    griddep_launch();
    const float* a = p.a + (int64_t)r * p.d;
    bool bad = false;
    if (p.a_row) {
        const int32_t idx = p.a_row[r];
        bad = idx < 0 || idx >= p.a_rows;  // an out-of-range token: flag it and write nothing
        a = p.a + (int64_t)(bad ? 0 : idx) * p.d;
        if (bad && t == 0 && crank == 0 && p.err) atomicOr(p.err, 1);
    }
    float s[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = j * NORM_THREADS + t;
        float v = 0.f;
        if (i < dl) {
            v = a[base + i];
            if (p.b) v = v + p.b[(int64_t)r * p.d + base + i];
        }
        s[j] = v;
    }
    F2 ss = f2_two_prod(s[0], s[0]);
#pragma unroll
    for (int j = 1; j < PER; ++j) ss = f2_add(ss, f2_two_prod(s[j], s[j]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        ss = f2_add(ss, F2{__shfl_xor_sync(0xffffffffu, ss.hi, o), __shfl_xor_sync(0xffffffffu, ss.lo, o)});
    if (lane == 0) red[wid] = ss;
    __syncthreads();
    if (t == 0) {
        F2 v = red[0];
        for (int w = 1; w < NORM_THREADS / 32; ++w) v = f2_add(v, red[w]);
        part = v;
    }
    cluster.sync();
    if (t == 0) {
        F2 tot = *cluster.map_shared_rank(&part, 0);
        for (int c = 1; c < CL; ++c) tot = f2_add(tot, *cluster.map_shared_rank(&part, c));
        // mean of squares + eps: the pair divided by d (exact remainder by FMA), then eps added
        const float df = (float)p.d;
        const float qh = tot.hi / df;
        const float ql = (fmaf(-qh, df, tot.hi) + tot.lo) / df;
        inv_s = f2_rsqrt(f2_add(f2_quick(qh, ql), F2{p.eps, 0.f}));
    }
    cluster_arrive();  // this CTA is done reading the others' shared memory
    __syncthreads();
    const F2 inv = inv_s;
    if (!bad) {
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int i = j * NORM_THREADS + t;
            const bool in = i < dl;
            const int64_t gi = (int64_t)r * p.d + base + i;
            float y = 0.f;
            if (in) {
                if (p.sum) p.sum[gi] = s[j];
                y = f2_mul3_round(s[j], wv[j], inv);
                if (p.y) p.y[gi] = y;
            }
            // The block of 32 values lies in this warp's lanes (the slice is whole 32-value blocks when quantizing).
            if (p.yq && (j * NORM_THREADS + wid * 32) < dl) {
                float dsc;
                int8_t lv = 0;
                const int8_t qv = p.yl ? quantize2_lane(y, dsc, lv) : quantize_lane(y, dsc);
                if (in) {
                    p.yq[gi] = qv;
                    if (p.yl) p.yl[gi] = lv;
                }
                if (lane == 0) p.ys[gi / 32] = dsc;
            }
        }
    }
    cluster_wait();  // no CTA leaves while another may still read its shared memory
}

// One word per value, or with `l` the two-word form (high words to q, low words to l).
__global__ void __launch_bounds__(256) quantize_kernel(const float* __restrict__ x, int64_t nblocks,
                                                       int8_t* __restrict__ q, int8_t* __restrict__ l,
                                                       float* __restrict__ s) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t stride = (int64_t)gridDim.x * 8;
    for (int64_t b = warp; b < nblocks; b += stride) {
        float d;
        if (l) {
            int8_t lv;
            q[b * 32 + lane] = quantize2_lane(x[b * 32 + lane], d, lv);
            l[b * 32 + lane] = lv;
        } else {
            q[b * 32 + lane] = quantize_lane(x[b * 32 + lane], d);
        }
        if (lane == 0) s[b] = d;
    }
    griddep_launch();
}

}  // namespace

template <int PER, int CL>
cudaError_t launch_norm(const NormParams& p, int64_t rows, cudaStream_t st, int pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows * CL));
    cfg.blockDim = dim3(NORM_THREADS);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
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
    return cudaLaunchKernelEx(&cfg, add_rmsnorm_kernel<PER, CL>, p);
}

cudaError_t launch_add_rmsnorm(const NormCall& c, cudaStream_t st) {
    NormParams p = {c.a, c.a_row, c.a_rows, c.b, c.w, (int)c.d, c.eps, c.sum, c.y, c.yq, c.yl, c.ys, c.err, c.pf};
    // cluster size: up to 8 CTAs of at least 256 values each, each slice whole 32-value blocks
    int cl = 1;
    while (cl < 8 && c.d % (cl * 2 * 32) == 0 && c.d / (cl * 2) >= NORM_THREADS) cl *= 2;
    const int dl = (int)(c.d / cl);
    const int per = (dl + NORM_THREADS - 1) / NORM_THREADS;
#define Q8_NORM(CL)                                                                            \
    if (cl == CL) {                                                                            \
        if (per <= 1) return launch_norm<1, CL>(p, c.rows, st, c.pdl);                         \
        if (per <= 2) return launch_norm<2, CL>(p, c.rows, st, c.pdl);                         \
        if (per <= 4) return launch_norm<4, CL>(p, c.rows, st, c.pdl);                         \
        if (per <= 8) return launch_norm<8, CL>(p, c.rows, st, c.pdl);                         \
        if (per <= 16) return launch_norm<16, CL>(p, c.rows, st, c.pdl);                       \
        if (per <= NORM_MAX_D / NORM_THREADS) return launch_norm<32, CL>(p, c.rows, st, c.pdl); \
    }
    Q8_NORM(1)
    Q8_NORM(2)
    Q8_NORM(4)
    Q8_NORM(8)
#undef Q8_NORM
    return cudaErrorInvalidValue;
}

cudaError_t launch_quantize(const float* x, int64_t n, int8_t* q, float* s, cudaStream_t st, int8_t* l) {
    const int64_t nblocks = n / 32;
    int64_t grid = (nblocks + 7) / 8;
    const int64_t cap = (int64_t)device_info().sms * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    return launch(quantize_kernel, dim3((unsigned)grid), dim3(256), 0, st, 0, x, nblocks, q, l, s);
}

}  // namespace q8
