// Residual add + RMSNorm with the int8 epilogue, and the standalone activation quantizer.
//
// What it computes: forward_shim.rs module docs (a sum and the RMS norm of it as one row kernel writing the sum on; the
// activation a Q8_0 projection reads quantized in its producer's epilogue), ForwardShim::fits (AddNorm) and
// ForwardShim::supports (the residual summed in f32, uncompensated); lane_link.rs, Link::prim (Norm{x, add, w, rows,
// cols, eps}; the standalone Quant launch).
//
// How: one CTA per row (rows are at most a few thousand values and the kernel is latency-bound).  A warp holds 32
// consecutive values per step, so each 32-value quantisation block is one warp's registers and its maximum one warp
// reduction.  The mean of squares is summed in f64 and the norm factor taken in f64, so y is rounded to f32 once.
#include "common.cuh"
#include "kernels.h"

namespace q8 {
namespace {

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

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
    float* ys;
    int* err;
};

// PER values per thread (d <= PER * 256), kept in registers between the two passes.
template <int PER>
__global__ void __launch_bounds__(NORM_THREADS) add_rmsnorm_kernel(const NormParams p) {
    __shared__ double red[NORM_THREADS / 32];
    const int r = blockIdx.x;
    const int t = threadIdx.x;
    const int lane = t & 31, wid = t >> 5;
    griddep_wait();
    const float* a = p.a + (int64_t)r * p.d;
    if (p.a_row) {
        const int32_t idx = p.a_row[r];
        if (idx < 0 || idx >= p.a_rows) {  // an out-of-range token: flag it and write nothing
            if (t == 0 && p.err) atomicOr(p.err, 1);
            return;
        }
        a = p.a + (int64_t)idx * p.d;
    }
    float s[PER];
    double ss = 0.0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = j * NORM_THREADS + t;
        float v = 0.f;
        if (i < p.d) {
            v = a[i];
            if (p.b) v = v + p.b[(int64_t)r * p.d + i];
            ss = fma((double)v, (double)v, ss);
        }
        s[j] = v;
    }
    // f64 sum of squares over the row
    ss = group_sum<32>(ss);
    if (lane == 0) red[wid] = ss;
    __syncthreads();
    if (wid == 0) {
        double v = lane < NORM_THREADS / 32 ? red[lane] : 0.0;
        v = group_sum<32>(v);
        if (lane == 0) red[0] = v;
    }
    __syncthreads();
    const double inv = 1.0 / sqrt(red[0] / (double)p.d + (double)p.eps);
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = j * NORM_THREADS + t;
        const bool in = i < p.d;
        float y = 0.f;
        if (in) {
            if (p.sum) p.sum[(int64_t)r * p.d + i] = s[j];
            y = (float)((double)s[j] * inv * (double)p.w[i]);
            if (p.y) p.y[(int64_t)r * p.d + i] = y;
        }
        // The block of 32 values i0..i0+31 lies in this warp's lanes (d % 32 == 0 when quantizing).
        if (p.yq && (j * NORM_THREADS + wid * 32) < p.d) {
            float dsc;
            const int8_t qv = quantize_lane(y, dsc);
            if (in) p.yq[(int64_t)r * p.d + i] = qv;
            if (lane == 0) p.ys[((int64_t)r * p.d + i) / 32] = dsc;
        }
    }
    griddep_launch();
}

__global__ void __launch_bounds__(256) quantize_kernel(const float* __restrict__ x, int64_t nblocks,
                                                       int8_t* __restrict__ q, float* __restrict__ s) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t stride = (int64_t)gridDim.x * 8;
    for (int64_t b = warp; b < nblocks; b += stride) {
        float d;
        const int8_t v = quantize_lane(x[b * 32 + lane], d);
        q[b * 32 + lane] = v;
        if (lane == 0) s[b] = d;
    }
    griddep_launch();
}

}  // namespace

cudaError_t launch_add_rmsnorm(const NormCall& c, cudaStream_t st) {
    NormParams p = {c.a, c.a_row, c.a_rows, c.b, c.w, (int)c.d, c.eps, c.sum, c.y, c.yq, c.ys, c.err};
    const dim3 grid((unsigned)c.rows), block(NORM_THREADS);
    const int per = (int)((c.d + NORM_THREADS - 1) / NORM_THREADS);
    if (per <= 1) return launch(add_rmsnorm_kernel<1>, grid, block, 0, st, c.pdl, p);
    if (per <= 2) return launch(add_rmsnorm_kernel<2>, grid, block, 0, st, c.pdl, p);
    if (per <= 4) return launch(add_rmsnorm_kernel<4>, grid, block, 0, st, c.pdl, p);
    if (per <= 8) return launch(add_rmsnorm_kernel<8>, grid, block, 0, st, c.pdl, p);
    if (per <= 16) return launch(add_rmsnorm_kernel<16>, grid, block, 0, st, c.pdl, p);
    if (per <= NORM_MAX_D / NORM_THREADS) return launch(add_rmsnorm_kernel<32>, grid, block, 0, st, c.pdl, p);
    return cudaErrorInvalidValue;
}

cudaError_t launch_quantize(const float* x, int64_t n, int8_t* q, float* s, cudaStream_t st) {
    const int64_t nblocks = n / 32;
    int64_t grid = (nblocks + 7) / 8;
    const int64_t cap = (int64_t)device_info().sms * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    return launch(quantize_kernel, dim3((unsigned)grid), dim3(256), 0, st, 0, x, nblocks, q, s);
}

}  // namespace q8
