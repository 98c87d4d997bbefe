// The C ABI of q8moe.h: argument checks (refusal by name, as kernel_refusal in forward_shim.rs and LaneError in
// lane/mod.rs refuse), the workspace, and the per-operation entry points.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "kernels.h"
#include "q8moe.h"

namespace q8 {

extern int kDenseMmaMinRows;    // gemv.cu
extern int kGroupedMmaMinRows;  // moe_mma.cu
extern int kChunkAttnTensorCores;  // decode.cu
extern int kStreamedBatchAttention;  // decode.cu

static thread_local char g_err[512];

static int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

static int cuda_fail(cudaError_t e, const char* what) {
    return fail(Q8_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

const DeviceInfo& device_info() {
    static std::mutex mu;
    static std::vector<DeviceInfo> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1);
    DeviceInfo& d = cache[dev];
    if (d.sms == 0) {
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (d.sms <= 0) d.sms = 1;
    }
    return d;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

static int check_mat(const q8_mat* W, const char* name) {
    if (!W) return fail(Q8_EINVAL, "%s: null matrix", name);
    if (!W->q || !W->s) return fail(Q8_EINVAL, "%s: null quants or scales", name);
    if (W->rows < 1 || W->cols < 1) return fail(Q8_EINVAL, "%s: %lld x %lld", name, (long long)W->rows, (long long)W->cols);
    if (W->cols % 32) return fail(Q8_EUNSUPPORTED, "%s: %lld columns, not whole 32-value blocks", name, (long long)W->cols);
    if (W->cols > (1 << 20) || W->rows > (int64_t(1) << 30))
        return fail(Q8_EUNSUPPORTED, "%s: %lld x %lld is past the kernels' index range", name, (long long)W->rows,
                    (long long)W->cols);
    if (!aligned(W->q, 32)) return fail(Q8_EINVAL, "%s: quants not 32-byte aligned", name);
    if (!aligned(W->s, 4)) return fail(Q8_EINVAL, "%s: scales not 4-byte aligned", name);
    return Q8_OK;
}

// A quantized activation; `two`: the two-word form, whose low words must be given too.
static int check_act(const q8_act* a, const char* name, bool two = false) {
    if (!a || !a->q || !a->s) return fail(Q8_EINVAL, "%s: null quantized activation", name);
    if (!aligned(a->q, 32)) return fail(Q8_EINVAL, "%s: words not 32-byte aligned", name);
    if (!aligned(a->s, 4)) return fail(Q8_EINVAL, "%s: scales not 4-byte aligned", name);
    if (two && !a->lo) return fail(Q8_EINVAL, "%s: null low words (the two-word mode)", name);
    if (a->lo && !aligned(a->lo, 32)) return fail(Q8_EINVAL, "%s: low words not 32-byte aligned", name);
    return Q8_OK;
}

static bool valid_mode(q8_mode mode) { return mode == Q8_F32ACT_F64SUM || mode == Q8_INT8ACT || mode == Q8_INT8ACT2; }

// The same error reporting for the decode model (model.cu).
int model_fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

}  // namespace q8

using namespace q8;

struct q8_ws {
    char* scratch = nullptr;
    size_t bytes = 0;
    int* counters = nullptr;
    size_t n_counters = 0;
    Carve carve() const {
        Carve c;
        c.base = scratch;
        c.size = bytes;
        c.counters = counters;
        c.n_counters = n_counters;
        return c;
    }
};

static const size_t kDefaultScratch = size_t(64) << 20;
static const size_t kCounters = size_t(1) << 20;

extern "C" {

const char* q8_last_error(void) { return g_err; }

int q8_workspace_create(size_t bytes, q8_ws** ws) {
    g_err[0] = 0;
    if (!ws) return fail(Q8_EINVAL, "ws: null");
    *ws = nullptr;
    q8_ws* w = new q8_ws();
    w->bytes = bytes ? bytes : kDefaultScratch;
    w->n_counters = kCounters;
    cudaError_t e = cudaMalloc(&w->scratch, w->bytes);
    if (e == cudaSuccess) e = cudaMalloc(&w->counters, w->n_counters * sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(w->counters, 0, w->n_counters * sizeof(int));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(w->scratch);
        cudaFree(w->counters);
        delete w;
        return cuda_fail(e, "q8_workspace_create");
    }
    *ws = w;
    return Q8_OK;
}

void q8_workspace_destroy(q8_ws* ws) {
    if (!ws) return;
    cudaFree(ws->scratch);
    cudaFree(ws->counters);
    delete ws;
}

size_t q8_workspace_bytes(const q8_ws* ws) { return ws ? ws->bytes : 0; }

int q8_quantize(const float* x, int64_t rows, int64_t cols, const q8_act* out, q8_stream stream) {
    g_err[0] = 0;
    if (!x) return fail(Q8_EINVAL, "x: null");
    if (rows < 0 || cols < 0) return fail(Q8_EINVAL, "rows/cols negative");
    if (cols % 32) return fail(Q8_EUNSUPPORTED, "cols %lld: not whole 32-value blocks", (long long)cols);
    if (int r = check_act(out, "out")) return r;
    if (rows * cols == 0) return Q8_OK;
    cudaError_t e = launch_quantize(x, rows * cols, out->q, out->s, (cudaStream_t)stream, out->lo);
    return e == cudaSuccess ? Q8_OK : cuda_fail(e, "q8_quantize");
}

int add_rmsnorm_q8(const float* a, const float* b, const float* w, int64_t rows, int64_t d, float eps, float* sum_out,
                   float* y_out, const q8_act* yq, q8_stream stream) {
    g_err[0] = 0;
    if (!a || !w) return fail(Q8_EINVAL, "a or w: null");
    if (rows < 0 || d < 1) return fail(Q8_EINVAL, "rows %lld, d %lld", (long long)rows, (long long)d);
    if (d > 8192) return fail(Q8_EUNSUPPORTED, "d %lld: a row kernel holds at most 8192 values", (long long)d);
    if (!(eps >= 0.f)) return fail(Q8_EINVAL, "eps: negative or NaN");
    if (!sum_out && !y_out && !yq) return fail(Q8_EINVAL, "no output requested");
    if (yq) {
        if (d % 32) return fail(Q8_EUNSUPPORTED, "d %lld: the int8 epilogue needs whole 32-value blocks", (long long)d);
        if (int r = check_act(yq, "yq")) return r;
    }
    if (rows == 0) return Q8_OK;
    if (rows > 0x7fffffff) return fail(Q8_EUNSUPPORTED, "rows: too many");
    NormCall c;
    c.a = a;
    c.b = b;
    c.w = w;
    c.rows = rows;
    c.d = d;
    c.eps = eps;
    c.sum = sum_out;
    c.y = y_out;
    c.yq = yq ? yq->q : nullptr;
    c.yl = yq ? yq->lo : nullptr;
    c.ys = yq ? yq->s : nullptr;
    cudaError_t e = launch_add_rmsnorm(c, (cudaStream_t)stream);
    return e == cudaSuccess ? Q8_OK : cuda_fail(e, "add_rmsnorm_q8");
}

// The projection's argument checks (no launch, no side effect).
static int gemv_check(const q8_mat* W, q8_mode mode, const float* x, const q8_act* xq, int64_t rows, float* y,
                      int32_t* dots) {
    if (int r = check_mat(W, "W")) return r;
    if (!valid_mode(mode)) return fail(Q8_EINVAL, "mode %d", (int)mode);
    if (rows < 0) return fail(Q8_EINVAL, "rows negative");
    if (rows > 65536) return fail(Q8_EUNSUPPORTED, "rows %lld: more activation rows than the kernel loops over",
                                  (long long)rows);
    if (!y && !dots) return fail(Q8_EINVAL, "y: null");
    if (mode == Q8_F32ACT_F64SUM && !x) return fail(Q8_EINVAL, "x: null (f32 mode reads x)");
    if (mode != Q8_F32ACT_F64SUM && !xq && !x) return fail(Q8_EINVAL, "xq and x: both null");
    if (xq && mode != Q8_F32ACT_F64SUM)
        if (int r = check_act(xq, "xq", mode == Q8_INT8ACT2)) return r;
    if (x && !aligned(x, 16)) return fail(Q8_EINVAL, "x: not 16-byte aligned");
    return Q8_OK;
}

static int gemv_common(const q8_mat* W, q8_mode mode, const float* x, const q8_act* xq, int64_t rows, float* y,
                       int32_t* dots, q8_ws* ws, cudaStream_t st, const char* who) {
    if (int r = gemv_check(W, mode, x, xq, rows, y, dots)) return r;
    if (rows == 0) return Q8_OK;
    Carve cv;
    if (ws) cv = ws->carve();
    GemvCall c;
    c.mode = (int)mode;
    c.k = W->cols;
    c.nseg = 1;
    c.seg[0].q = W->q;
    c.seg[0].s = W->s;
    c.seg[0].n = W->rows;
    c.seg[0].y = y;
    c.x = x;
    c.R = rows;
    c.dots = dots;
    if (dots && mode == Q8_INT8ACT2) c.dots_lo = dots + rows * W->rows * (W->cols / 32);
    if (mode != Q8_F32ACT_F64SUM) {
        if (xq) {
            c.xq = xq->q;
            c.xl = mode == Q8_INT8ACT2 ? xq->lo : nullptr;
            c.xs = xq->s;
        } else {
            if (!ws) return fail(Q8_EINVAL, "ws: null (x is quantized into workspace scratch)");
            int8_t* q = cv.take<int8_t>((size_t)(rows * W->cols));
            float* s = cv.take<float>((size_t)(rows * W->cols / 32));
            int8_t* l = mode == Q8_INT8ACT2 ? cv.take<int8_t>((size_t)(rows * W->cols)) : nullptr;
            if (cv.overflow) return fail(Q8_ENOSPACE, "%s: workspace too small for the quantized activation", who);
            cudaError_t e = launch_quantize(x, rows * W->cols, q, s, st, l);
            if (e != cudaSuccess) return cuda_fail(e, who);
            c.xq = q;
            c.xl = l;
            c.xs = s;
        }
    }
    size_t need = 0, cnt = 0;
    gemv_scratch(c, &need, &cnt);
    if ((need || cnt) && !ws) return fail(Q8_EINVAL, "ws: null (this shape is cut along k)");
    cudaError_t e = launch_gemv(c, cv, st);
    if (cv.overflow) return fail(Q8_ENOSPACE, "%s: workspace too small (%zu bytes, %zu counters needed)", who, need, cnt);
    return e == cudaSuccess ? Q8_OK : cuda_fail(e, who);
}

int q8_gemv(const q8_mat* W, q8_mode mode, const float* x, const q8_act* xq, int64_t rows, float* y, q8_ws* ws,
            q8_stream stream) {
    g_err[0] = 0;
    if (!y) return fail(Q8_EINVAL, "y: null");
    return gemv_common(W, mode, x, xq, rows, y, nullptr, ws, (cudaStream_t)stream, "q8_gemv");
}

int q8_gemv_blockdots(const q8_mat* W, const q8_act* xq, int64_t rows, int32_t* dots, float* y, q8_ws* ws,
                      q8_stream stream) {
    g_err[0] = 0;
    if (!dots || !y) return fail(Q8_EINVAL, "dots or y: null");
    if (!xq) return fail(Q8_EINVAL, "xq: null");
    return gemv_common(W, xq->lo ? Q8_INT8ACT2 : Q8_INT8ACT, nullptr, xq, rows, y, dots, ws, (cudaStream_t)stream,
                       "q8_gemv_blockdots");
}

static int check_plan(const q8_moe_plan* plan) {
    if (!plan->counts || !plan->offsets || !plan->lists || !plan->active) return fail(Q8_EINVAL, "plan: null array");
    return Q8_OK;
}

int moe_route_topk(const q8_mat* router, q8_mode mode, const float* x, const q8_act* xq, int64_t rows, int k,
                   int32_t* ids, float* gates, float* logits, const q8_moe_plan* plan, q8_ws* ws, q8_stream stream) {
    g_err[0] = 0;
    if (int r = check_mat(router, "router")) return r;
    const int64_t E = router->rows;
    if (k < 1 || k > 32) return fail(Q8_EUNSUPPORTED, "k %d: the router keeps 1 to 32 experts", k);
    if (E > 8192) return fail(Q8_EUNSUPPORTED, "%lld experts: at most 8192", (long long)E);
    if (k > E) return fail(Q8_EINVAL, "k %d above the %lld experts", k, (long long)E);
    if (!ids || !gates) return fail(Q8_EINVAL, "ids or gates: null");
    if (!ws) return fail(Q8_EINVAL, "ws: null");
    if (rows < 0) return fail(Q8_EINVAL, "rows negative");
    if (rows * k > 65536) return fail(Q8_EUNSUPPORTED, "rows*k %lld: the grouping handles at most 65536 choices",
                                      (long long)(rows * k));
    if (plan)
        if (int r = check_plan(plan)) return r;
    if (rows == 0) return Q8_OK;
    cudaStream_t st = (cudaStream_t)stream;
    if (!valid_mode(mode)) return fail(Q8_EINVAL, "mode %d", (int)mode);
    const bool act = mode != Q8_F32ACT_F64SUM ? (xq && !check_act(xq, "xq", mode == Q8_INT8ACT2))
                                              : (x && aligned(x, 16));
    if (rows == 1 && !plan && act && route_row_supported((int)mode, E, router->cols, k)) {
        // one row: the projection and the top-k in one cluster launch
        RouteRowCall c;
        c.mode = (int)mode;
        c.q = router->q;
        c.s = router->s;
        c.E = E;
        c.d = router->cols;
        c.K = k;
        c.x = x;
        c.xq = mode != Q8_F32ACT_F64SUM ? xq->q : nullptr;
        c.xl = mode == Q8_INT8ACT2 ? xq->lo : nullptr;
        c.xs = mode != Q8_F32ACT_F64SUM ? xq->s : nullptr;
        c.logits = logits;
        c.ids = ids;
        c.gates = gates;
        cudaError_t e = launch_route_row(c, st);
        return e == cudaSuccess ? Q8_OK : cuda_fail(e, "moe_route_topk");
    }
    q8_ws tmp = *ws;
    float* l = logits;
    Carve cv = ws->carve();
    if (!l) {
        l = cv.take<float>((size_t)(rows * E));
        if (cv.overflow) return fail(Q8_ENOSPACE, "moe_route_topk: workspace too small for the logits");
        tmp.scratch = ws->scratch + cv.used;
        tmp.bytes = ws->bytes - cv.used;
    }
    int* done = nullptr;  // the top-k's arrival counter: the workspace's last one, kept from the projection
    if (plan && tmp.n_counters > 0) {
        done = tmp.counters + tmp.n_counters - 1;
        tmp.n_counters -= 1;
    }
    int r = gemv_common(router, mode, x, xq, rows, l, nullptr, &tmp, st, "moe_route_topk");
    if (r) return r;
    TopkCall t;
    t.done = done;
    t.logits = l;
    t.R = rows;
    t.E = E;
    t.K = k;
    t.ids = ids;
    t.gates = gates;
    if (plan) {
        t.plan.counts = plan->counts;
        t.plan.offsets = plan->offsets;
        t.plan.lists = plan->lists;
        t.plan.active = plan->active;
    }
    cudaError_t e = launch_topk(t, st);
    return e == cudaSuccess ? Q8_OK : cuda_fail(e, "moe_route_topk");
}

}  // extern "C"

extern "C" {

// A shared expert's shapes: gate and up [sdff][d], down [d][sdff], whole 32-value blocks.
static int check_shared(const q8_shared_expert* sh, int64_t d, int64_t* sdff) {
    *sdff = 0;
    if (!sh) return Q8_OK;
    if (int r = check_mat(&sh->gate, "shared.gate")) return r;
    if (int r = check_mat(&sh->up, "shared.up")) return r;
    if (int r = check_mat(&sh->down, "shared.down")) return r;
    const int64_t f = sh->gate.rows;
    if (sh->up.rows != f || sh->gate.cols != d || sh->up.cols != d || sh->down.rows != d || sh->down.cols != f)
        return fail(Q8_EINVAL, "shared: gate/up must be [sdff, %lld] and down [%lld, sdff]", (long long)d, (long long)d);
    *sdff = f;
    return Q8_OK;
}

int moe_gate_up(const q8_mat* gate, const q8_mat* up, int64_t dff, q8_mode mode, const float* x, const q8_act* xq,
                int64_t rows, int k, const int32_t* ids, const q8_moe_plan* plan, float* h, const q8_act* hq,
                const q8_shared_expert* shared, q8_ws* ws, q8_stream stream) {
    g_err[0] = 0;
    if (int r = check_mat(gate, "gate")) return r;
    if (int r = check_mat(up, "up")) return r;
    if (gate->rows != up->rows || gate->cols != up->cols) return fail(Q8_EINVAL, "gate and up differ in shape");
    if (dff < 1 || gate->rows % dff) return fail(Q8_EINVAL, "dff %lld does not divide the %lld stacked rows",
                                                (long long)dff, (long long)gate->rows);
    if (!valid_mode(mode)) return fail(Q8_EINVAL, "mode %d", (int)mode);
    if (k < 1 || k > 32) return fail(Q8_EUNSUPPORTED, "k %d: 1 to 32 experts a row", k);
    if (!ids || !h || !ws) return fail(Q8_EINVAL, "ids, h or ws: null");
    if (rows < 0) return fail(Q8_EINVAL, "rows negative");
    if (rows > 1 && !plan) return fail(Q8_EINVAL, "plan: null (a chunk of %lld rows is grouped by expert)", (long long)rows);
    if (mode == Q8_F32ACT_F64SUM && (!x || !aligned(x, 16))) return fail(Q8_EINVAL, "x: null or not 16-byte aligned");
    if (mode != Q8_F32ACT_F64SUM) {
        if (int r = check_act(xq, "xq", mode == Q8_INT8ACT2)) return r;
        if (hq)
            if (int r = check_act(hq, "hq", mode == Q8_INT8ACT2)) return r;
        if (dff % 32) return fail(Q8_EUNSUPPORTED, "dff %lld: the int8 epilogue needs whole 32-row blocks", (long long)dff);
    }
    if (!experts_supported((int)mode, gate->cols))
        return fail(Q8_EUNSUPPORTED, "d %lld: an expert row wider than one pass of the kernel", (long long)gate->cols);
    if (plan)
        if (int r = check_plan(plan)) return r;
    int64_t sdff = 0;
    if (int r = check_shared(shared, gate->cols, &sdff)) return r;
    if (rows == 0) return Q8_OK;
    cudaStream_t st = (cudaStream_t)stream;
    ExpertCall c;
    c.mode = (int)mode;
    c.q0 = gate->q;
    c.s0 = gate->s;
    c.q1 = up->q;
    c.s1 = up->s;
    if (shared) {
        c.sq0 = shared->gate.q;
        c.ss0 = shared->gate.s;
        c.sq1 = shared->up.q;
        c.ss1 = shared->up.s;
        c.sdff = sdff;
    }
    c.E = gate->rows / dff;
    c.out_rows = dff;
    c.k = gate->cols;
    c.R = rows;
    c.K = k;
    c.ids = ids;
    c.x = x;
    c.xq = mode != Q8_F32ACT_F64SUM ? xq->q : nullptr;
    c.xl = mode == Q8_INT8ACT2 ? xq->lo : nullptr;
    c.xs = mode != Q8_F32ACT_F64SUM ? xq->s : nullptr;
    c.h = h;
    if (plan) {
        c.plan.counts = plan->counts;
        c.plan.offsets = plan->offsets;
        c.plan.lists = plan->lists;
        c.plan.active = plan->active;
    }
    if (mode != Q8_F32ACT_F64SUM && hq && gate_row_supported(c)) {  // one row: the kernel quantizes each 32-row block
        c.hq_out = hq->q;
        c.hl_out = mode == Q8_INT8ACT2 ? hq->lo : nullptr;
        c.hs_out = hq->s;
    }
    Carve cv = ws->carve();
    cudaError_t e = launch_gate_up(c, cv, st);
    if (cv.overflow) return fail(Q8_ENOSPACE, "moe_gate_up: workspace too small for the int8 epilogue's counters");
    if (e == cudaSuccess && mode != Q8_F32ACT_F64SUM && hq && !c.hq_out)
        e = launch_quantize(h, rows * k * dff + rows * sdff, hq->q, hq->s, st, mode == Q8_INT8ACT2 ? hq->lo : nullptr);
    return e == cudaSuccess ? Q8_OK : cuda_fail(e, "moe_gate_up");
}

int moe_down_combine(const q8_mat* down, int64_t d, q8_mode mode, const float* h, const q8_act* hq, int64_t rows,
                     int k, const int32_t* ids, const float* gates, const q8_moe_plan* plan, const float* residual,
                     float* y, float* expert_out, const q8_shared_expert* shared, q8_ws* ws, q8_stream stream) {
    g_err[0] = 0;
    if (int r = check_mat(down, "down")) return r;
    if (d < 1 || down->rows % d) return fail(Q8_EINVAL, "d %lld does not divide the %lld stacked rows", (long long)d,
                                            (long long)down->rows);
    if (!valid_mode(mode)) return fail(Q8_EINVAL, "mode %d", (int)mode);
    if (k < 1 || k > 32) return fail(Q8_EUNSUPPORTED, "k %d: 1 to 32 experts a row", k);
    if (!ids || !gates || !y || !ws) return fail(Q8_EINVAL, "ids, gates, y or ws: null");
    if (rows < 0) return fail(Q8_EINVAL, "rows negative");
    if (rows > 1 && !plan) return fail(Q8_EINVAL, "plan: null (a chunk of %lld rows is grouped by expert)", (long long)rows);
    if (mode == Q8_F32ACT_F64SUM && (!h || !aligned(h, 16))) return fail(Q8_EINVAL, "h: null or not 16-byte aligned");
    if (mode != Q8_F32ACT_F64SUM) {
        if (hq) {
            if (int r = check_act(hq, "hq", mode == Q8_INT8ACT2)) return r;
        } else if (!h || !aligned(h, 16)) {
            return fail(Q8_EINVAL, "hq and h: both null (or h not 16-byte aligned)");
        }
    }
    if (!experts_supported((int)mode, down->cols))
        return fail(Q8_EUNSUPPORTED, "dff %lld: an expert row wider than one pass of the kernel", (long long)down->cols);
    if (plan)
        if (int r = check_plan(plan)) return r;
    int64_t sdff = 0;
    if (int r = check_shared(shared, d, &sdff)) return r;
    if (rows == 0) return Q8_OK;
    cudaStream_t st = (cudaStream_t)stream;
    ExpertCall c;
    c.mode = (int)mode;
    c.q0 = down->q;
    c.s0 = down->s;
    if (shared) {
        c.sq0 = shared->down.q;
        c.ss0 = shared->down.s;
        c.sdff = sdff;
    }
    c.E = down->rows / d;
    c.out_rows = d;
    c.k = down->cols;
    c.R = rows;
    c.K = k;
    c.ids = ids;
    c.gates = gates;
    c.x = h;
    if (mode != Q8_F32ACT_F64SUM && hq) {
        c.x = nullptr;
        c.xq = hq->q;
        c.xl = mode == Q8_INT8ACT2 ? hq->lo : nullptr;
        c.xs = hq->s;
    }
    c.residual = residual;
    c.y = y;
    c.expert_out = expert_out;
    if (plan) {
        c.plan.counts = plan->counts;
        c.plan.offsets = plan->offsets;
        c.plan.lists = plan->lists;
        c.plan.active = plan->active;
    }
    Carve cv = ws->carve();
    if (mode != Q8_F32ACT_F64SUM && !hq && (rows > 1 || plan)) {  // a chunk reads its hidden rows quantized
        const int64_t nh = rows * k * down->cols + rows * sdff;  // the routed hidden rows, then the shared expert's
        int8_t* q = cv.take<int8_t>((size_t)nh);
        float* s = cv.take<float>((size_t)(nh / 32));
        int8_t* l = mode == Q8_INT8ACT2 ? cv.take<int8_t>((size_t)nh) : nullptr;
        if (cv.overflow) return fail(Q8_ENOSPACE, "moe_down_combine: workspace too small for the quantized rows");
        cudaError_t qe = launch_quantize(h, nh, q, s, st, l);
        if (qe != cudaSuccess) return cuda_fail(qe, "moe_down_combine");
        c.x = nullptr;
        c.xq = q;
        c.xl = l;
        c.xs = s;
    }
    size_t need = 0, cnt = 0;
    down_scratch(c, &need, &cnt);
    cudaError_t e = launch_down_combine(c, cv, st);
    if (cv.overflow) return fail(Q8_ENOSPACE, "moe_down_combine: workspace too small (%zu bytes, %zu counters)", need, cnt);
    return e == cudaSuccess ? Q8_OK : cuda_fail(e, "moe_down_combine");
}

int q8_set_tensor_core_rows(int rows) {
    g_err[0] = 0;
    if (rows != 0 && rows != -1 && (rows < 16 || rows > 64))
        return fail(Q8_EINVAL, "rows %d: -1 (automatic), 0 (off) or 16 to 64", rows);
    kDenseMmaMinRows = rows;
    return Q8_OK;
}

int q8_set_grouped_tensor_core_rows(int rows) {
    g_err[0] = 0;
    if (rows != 0 && (rows < 16 || rows > 64)) return fail(Q8_EINVAL, "rows %d: 0 (off) or 16 to 64", rows);
    kGroupedMmaMinRows = rows;
    return Q8_OK;
}

int q8_set_persistent_decode(int on) {
    g_err[0] = 0;
    if (on != 0 && on != 1) return fail(Q8_EINVAL, "on %d: 0 or 1", on);
    kPersistentDecode = on;
    return Q8_OK;
}

int q8_set_streamed_batch_attention(int min_batch) {
    g_err[0] = 0;
    if (min_batch != 0 && min_batch < 2) return fail(Q8_EINVAL, "min_batch %d: 0 or at least 2", min_batch);
    kStreamedBatchAttention = min_batch;
    return Q8_OK;
}

int q8_set_tensor_core_attention(int on) {
    g_err[0] = 0;
    if (on != 0 && on != 1) return fail(Q8_EINVAL, "on %d: 0 or 1", on);
    kChunkAttnTensorCores = on;
    return Q8_OK;
}

int moe_route_topk_f32(const float* router, int64_t E, int64_t d, const float* x, int64_t rows, int k, int32_t* ids,
                       float* gates, float* logits, const q8_moe_plan* plan, q8_ws* ws, q8_stream stream) {
    g_err[0] = 0;
    if (!router || !x) return fail(Q8_EINVAL, "router or x: null");
    if (!aligned(router, 16) || !aligned(x, 16)) return fail(Q8_EINVAL, "router or x: not 16-byte aligned");
    if (E < 1 || d < 1) return fail(Q8_EINVAL, "experts %lld, d %lld", (long long)E, (long long)d);
    if (d % 32) return fail(Q8_EUNSUPPORTED, "d %lld: not whole 32-value blocks", (long long)d);
    if (k < 1 || k > 32) return fail(Q8_EUNSUPPORTED, "k %d: the router keeps 1 to 32 experts", k);
    if (E > 8192) return fail(Q8_EUNSUPPORTED, "%lld experts: at most 8192", (long long)E);
    if (k > E) return fail(Q8_EINVAL, "k %d above the %lld experts", k, (long long)E);
    if (!ids || !gates || !ws) return fail(Q8_EINVAL, "ids, gates or ws: null");
    if (rows < 0) return fail(Q8_EINVAL, "rows negative");
    if (rows * k > 65536) return fail(Q8_EUNSUPPORTED, "rows*k %lld: the grouping handles at most 65536 choices",
                                      (long long)(rows * k));
    if (plan)
        if (int r = check_plan(plan)) return r;
    if (rows == 0) return Q8_OK;
    cudaStream_t st = (cudaStream_t)stream;
    Carve cv = ws->carve();
    float* l = logits ? logits : cv.take<float>((size_t)(rows * E));
    if (cv.overflow) return fail(Q8_ENOSPACE, "moe_route_topk_f32: workspace too small for the logits");
    cudaError_t e = launch_router_f32(router, E, d, x, rows, l, 0, st);
    if (e != cudaSuccess) return cuda_fail(e, "moe_route_topk_f32");
    TopkCall t;
    t.done = plan && ws->n_counters > 0 ? ws->counters + ws->n_counters - 1 : nullptr;
    t.logits = l;
    t.R = rows;
    t.E = E;
    t.K = k;
    t.ids = ids;
    t.gates = gates;
    if (plan) {
        t.plan.counts = plan->counts;
        t.plan.offsets = plan->offsets;
        t.plan.lists = plan->lists;
        t.plan.active = plan->active;
    }
    e = launch_topk(t, st);
    return e == cudaSuccess ? Q8_OK : cuda_fail(e, "moe_route_topk_f32");
}

}  // extern "C"

namespace q8 {

Carve workspace_carve(const q8_ws* ws) { return ws->carve(); }

// Scratch one q8_gemv call takes (bytes and arrival counters): the quantized activation when x is quantized inside
// the call, then the partial sums of a projection cut along k; each region rounded up to 256 bytes as a workspace
// carve rounds it.
void gemv_call_scratch(const q8_mat* W, q8_mode mode, const float* x, const q8_act* xq, int64_t rows, size_t* bytes,
                       size_t* counters) {
    GemvCall c;  // the call q8_gemv would launch, so that the path chosen (bulk-copied rows or not) is the same
    c.mode = (int)mode;
    c.k = W->cols;
    c.nseg = 1;
    c.seg[0].q = W->q;
    c.seg[0].s = W->s;
    c.seg[0].n = W->rows;
    c.x = x;
    c.R = rows;
    size_t b = 0;
    auto region = [&](size_t n) { b = ((b + 255) & ~size_t(255)) + n; };
    if (mode != Q8_F32ACT_F64SUM && !xq) {  // the quantized activation: words, scales (and low words)
        region((size_t)(rows * W->cols));
        region((size_t)(rows * W->cols / 32) * sizeof(float));
        if (mode == Q8_INT8ACT2) region((size_t)(rows * W->cols));
    }
    size_t pb = 0, pc = 0;
    gemv_scratch(c, &pb, &pc);
    if (pb) region(pb);
    *bytes = b;
    *counters = pc;
}

// q8_gemv over scratch memory the caller already holds instead of a workspace.  Every argument is checked first; when
// they pass, the first `zero_counters` counters (those the call will use) are cleared on `st` before the launch, so a
// call starts from zero even if an earlier one was cut short.
int gemv_over_scratch(const q8_mat* W, q8_mode mode, const float* x, const q8_act* xq, int64_t rows, float* y,
                      char* scratch, size_t bytes, int* counters, size_t n_counters, size_t zero_counters,
                      cudaStream_t st, const char* who) {
    g_err[0] = 0;
    if (!y) return fail(Q8_EINVAL, "y: null");
    if (int r = gemv_check(W, mode, x, xq, rows, y, nullptr)) return r;
    if (rows == 0) return Q8_OK;
    if (zero_counters) {
        cudaError_t e = cudaMemsetAsync(counters, 0, zero_counters * sizeof(int), st);
        if (e != cudaSuccess) return cuda_fail(e, who);
    }
    q8_ws w;
    w.scratch = scratch;
    w.bytes = bytes;
    w.counters = counters;
    w.n_counters = n_counters;
    return gemv_common(W, mode, x, xq, rows, y, nullptr, &w, st, who);
}

}  // namespace q8
