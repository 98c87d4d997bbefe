// Internal launch interface between the C ABI (api.cu) and the kernel files.  Host code only.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "prefetch.h"
#include "q8moe.h"

namespace q8 {

// Device facts the launchers size grids by (cached per device).
struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;
};
const DeviceInfo& device_info();

// A bump allocator over one workspace's scratch and counters, for the launches of one call.
struct Carve {
    char* base = nullptr;
    size_t size = 0, used = 0;
    int* counters = nullptr;
    size_t n_counters = 0, used_counters = 0;
    bool overflow = false;
    template <typename T>
    T* take(size_t n) {
        size_t off = (used + 255) & ~size_t(255);
        size_t bytes = n * sizeof(T);
        if (off + bytes > size) {
            overflow = true;
            return nullptr;
        }
        used = off + bytes;
        return reinterpret_cast<T*>(base + off);
    }
    int* take_counters(size_t n) {
        if (used_counters + n > n_counters) {
            overflow = true;
            return nullptr;
        }
        int* p = counters + used_counters;
        used_counters += n;
        return p;
    }
};

// ---- projections ------------------------------------------------------------------------------------------------
// One matrix of a (possibly merged) projection: all segments share cols and the activation.
struct GemvSeg {
    const int8_t* q = nullptr;
    const float* s = nullptr;
    int64_t n = 0;
    float* y = nullptr;                  // [R][n]
    const float* residual = nullptr;     // optional: y = fl32(residual + fl32(acc))
};

struct GemvCall {
    int mode = 0;
    int64_t k = 0;
    int nseg = 1;
    GemvSeg seg[3];
    const float* x = nullptr;            // [R][k] (mode 0)
    const int8_t* xq = nullptr;          // [R][k] (modes 1 and 2: the words; in mode 2 the high words)
    const int8_t* xl = nullptr;          // [R][k] (mode 2: the low words)
    const float* xs = nullptr;           // [R][k/32]
    int64_t R = 1;
    int32_t* dots = nullptr;             // modes 1, 2 debug export [R][n][k/32] (single segment; mode 2: high words)
    int32_t* dots_lo = nullptr;          // mode 2 debug export of the low words' dots
    int* err = nullptr;                  // device error word for a pipeline wait that gave up
    L2Prefetch pf;                       // weights of later launches to fetch into L2 at the start
    int pdl = 0;                         // launch with programmatic dependent launch allowed
    // optional RMSNorm prologue (one row, k a multiple of 256 and at most 4096): x = RMSNorm(norm_a) * norm_w formed
    // inside the launch; with norm_a_row the row is norm_a + (*norm_a_row) * k (an embedding gather; bit 1 of err
    // for an index outside [0, norm_a_rows)) and the gathered row is written to norm_sum_out
    const float* norm_a = nullptr;
    const int32_t* norm_a_row = nullptr;
    int64_t norm_a_rows = 0;
    const float* norm_w = nullptr;
    float eps = 0.f;
    float* norm_sum_out = nullptr;
};
bool gemv_norm_supported(const GemvCall& c);

// Scratch needed by a projection (bytes, counters).
void gemv_scratch(const GemvCall& c, size_t* bytes, size_t* counters);
cudaError_t launch_gemv(const GemvCall& c, Carve& ws, cudaStream_t st);

// ---- norm and quantisation ------------------------------------------------------------------------------------
struct NormCall {
    const float* a = nullptr;
    const int32_t* a_row = nullptr;      // optional: a's row for each row r is a + a_row[r]*d (an embedding gather)
    int64_t a_rows = 0;                  // rows of the gathered table (bounds check)
    const float* b = nullptr;
    const float* w = nullptr;
    int64_t rows = 0, d = 0;
    float eps = 0.f;
    float* sum = nullptr;
    float* y = nullptr;
    int8_t* yq = nullptr;
    int8_t* yl = nullptr;                // with yq: the two-word form's low words
    float* ys = nullptr;
    int* err = nullptr;                  // device error word for a gathered row out of range
    L2Prefetch pf;                       // weights of later launches to fetch into L2 at the start
    int pdl = 0;
};
cudaError_t launch_add_rmsnorm(const NormCall& c, cudaStream_t st);
// One word per value, or with l the two-word form (high words to q, low words to l).
cudaError_t launch_quantize(const float* x, int64_t n, int8_t* q, float* s, cudaStream_t st, int8_t* l = nullptr);

// ---- mixture ----------------------------------------------------------------------------------------------------
struct PlanPtrs {
    int32_t* counts = nullptr;    // [E]
    int32_t* offsets = nullptr;   // [E+1]
    int32_t* lists = nullptr;     // [R*K]
    int32_t* active = nullptr;    // [E+1]: count then the active experts ascending
};

// The stacked expert matrices whose chosen rows the top-k kernel prefetches into L2 once it has chosen (one row).
struct ExpertPrefetch {
    const int8_t* gq = nullptr;
    const float* gs = nullptr;
    const int8_t* uq = nullptr;
    const float* us = nullptr;
    const int8_t* dq = nullptr;
    const float* ds = nullptr;
    int64_t dff = 0, d = 0;
};

struct TopkCall {
    ExpertPrefetch xp;
    const float* logits = nullptr;  // [R][E]
    int64_t R = 1, E = 0;
    int K = 0;
    int32_t* ids = nullptr;
    float* gates = nullptr;
    PlanPtrs plan;                  // filled when plan.counts != nullptr
    int* done = nullptr;            // with a plan: one zero-at-rest counter, so that several CTAs can take the rows
    L2Prefetch pf;                       // weights of later launches to fetch into L2 at the start
    int pdl = 0;
};
cudaError_t launch_topk(const TopkCall& c, cudaStream_t st);

// A router of f32 values (lane_link.rs, Link::prim: Router::F32): logits[r][e] = w[e] . x[r], f32 products summed per
// 32 values and then in f64.
cudaError_t launch_router_f32(const float* w, int64_t E, int64_t d, const float* x, int64_t R, float* logits,
                              int pdl, cudaStream_t st);

struct ExpertCall {
    int mode = 0;
    // gate-up: w0 = gate, w1 = up (rows E*dff, cols d); down: w0 = down (rows E*d, cols dff)
    const int8_t* q0 = nullptr;
    const float* s0 = nullptr;
    const int8_t* q1 = nullptr;
    const float* s1 = nullptr;
    int64_t E = 0, out_rows = 0, k = 0;  // out_rows per expert (dff for gate-up, d for down); k = input width
    int64_t R = 1;
    int K = 0;
    const int32_t* ids = nullptr;
    const float* gates = nullptr;
    PlanPtrs plan;                       // used when plan.active != nullptr, else choice j is group j (R == 1)
    const float* x = nullptr;            // gate-up: x [R][k]; down: h [R*K][k] (f32; for one row in mode 1 the kernel
                                         // quantizes it as it stages it)
    const int8_t* xq = nullptr;          // modes 1, 2: gate-up xq [R][k]; down hq [R*K][k]
    const int8_t* xl = nullptr;          // mode 2: the low words beside xq
    const float* xs = nullptr;
    float* h = nullptr;                  // gate-up out [R*K][dff]
    int8_t* hq_out = nullptr;            // gate-up, one row, int8 modes: h quantized per 32 rows (dff % 32 == 0)
    int8_t* hl_out = nullptr;            //   (mode 2: its low words)
    float* hs_out = nullptr;             //   and its scales [K][dff/32]
    const float* residual = nullptr;     // down
    float* y = nullptr;                  // down out [R][d]
    float* expert_out = nullptr;         // down out [R][K][d]
    // a shared expert every row passes through, unweighted (sdff > 0): gate-up takes sq0/ss0 = its gate and sq1/ss1 =
    // its up [sdff][k], and writes its hidden rows after the routed ones (h + R*K*out_rows, [R][sdff]; the int8 forms
    // likewise); down takes sq0/ss0 = its down [out_rows][sdff] and reads those hidden rows
    const int8_t* sq0 = nullptr;
    const float* ss0 = nullptr;
    const int8_t* sq1 = nullptr;
    const float* ss1 = nullptr;
    int64_t sdff = 0;
    int* err = nullptr;                  // device error word for a pipeline wait that gave up
    L2Prefetch pf;                       // weights of later launches to fetch into L2 at the start
    int pdl = 0;
};
void gate_up_scratch(const ExpertCall& c, size_t* bytes, size_t* counters);
void down_scratch(const ExpertCall& c, size_t* bytes, size_t* counters);
// The expert kernels read a whole row of k in one pass: k <= 4096 (int8 mode) or 3072 (f32 mode).
bool experts_supported(int mode, int64_t k);
cudaError_t launch_gate_up(const ExpertCall& c, Carve& ws, cudaStream_t st);
cudaError_t launch_down_combine(const ExpertCall& c, Carve& ws, cudaStream_t st);

// One token row (moe_row.cu): the router projection and its top-k in one cluster launch, and a down-and-combine that
// requests its weights before the dependency wait.
struct RouteRowCall {
    int mode = 0;
    const int8_t* q = nullptr;  // router [E][d]
    const float* s = nullptr;
    int64_t E = 0, d = 0;
    int K = 0;
    const float* x = nullptr;   // f32 mode
    const int8_t* xq = nullptr; // int8 modes
    const int8_t* xl = nullptr; // mode 2: the low words
    const float* xs = nullptr;
    float* logits = nullptr;    // optional [E]
    int32_t* ids = nullptr;
    float* gates = nullptr;
    // optional: the kernel forms x = RMSNorm(norm_a) * norm_w itself (d a multiple of 256, at most 4096) and writes it
    // to x_out (f32 mode) or xq_out / xs_out (int8 mode); x, xq and xs are then not read
    const float* norm_a = nullptr;
    const float* norm_w = nullptr;
    float eps = 0.f;
    float* x_out = nullptr;
    int8_t* xq_out = nullptr;
    int8_t* xl_out = nullptr;   // mode 2
    float* xs_out = nullptr;
    L2Prefetch pf;
    int pdl = 0;
};
bool route_row_supported(int mode, int64_t E, int64_t d, int K);
cudaError_t launch_route_row(const RouteRowCall& c, cudaStream_t st);
// Tensor-core products (moe_mma.cu) for a chunk's expert groups of nmin..moe_mma_max_rows() choices, int8 mode:
// gate-up (q1 set) writes h, down writes the per-choice outputs to `out`; other groups are left alone.  A chunk's
// groups take them from moe_mma_min_rows() rows on (q8_set_grouped_tensor_core_rows; moe_mma_grouped says whether a
// call has any to give), the CUDA-core kernels skipping those groups.
bool moe_mma_supported(const ExpertCall& c, bool dense = false);
bool moe_mma_grouped(const ExpertCall& c);
int moe_mma_min_rows();
int moe_mma_max_rows();
// dense_rows > 0: a dense projection of that many rows (E = K = 1, no plan: the rows are the one group)
cudaError_t launch_moe_mma(const ExpertCall& c, float* out, int max_groups, Carve& ws, cudaStream_t st,
                           const float* res = nullptr, int nmin = moe_mma_min_rows(), int dense_rows = 0);
// A dense int8-mode projection of 16..64 activation rows on the tensor cores (the grouped product with one group of
// every row; each segment's rows a multiple of 128, k a multiple of 128).
bool dense_mma_supported(const GemvCall& g);
cudaError_t launch_dense_mma(const GemvCall& g, Carve& ws, cudaStream_t st);
bool gate_row_supported(const ExpertCall& c);
cudaError_t launch_gate_row(const ExpertCall& c, Carve& ws, cudaStream_t st);
bool down_row_supported(const ExpertCall& c);
cudaError_t launch_down_row(const ExpertCall& c, cudaStream_t st);

// ---- decode-step pieces -----------------------------------------------------------------------------------------
struct AttnCall {
    // the projection's rows of this step, before QK-norm and RoPE: the kernel norms and turns them, appends k and v
    // at `pos` to the caches and attends rows 0..pos
    const float* q = nullptr;       // [heads][hd]
    const float* k = nullptr;       // [kv][hd]
    const float* v = nullptr;       // [kv][hd]
    const float* q_norm = nullptr;  // [hd], shared by the heads
    const float* k_norm = nullptr;
    const float* cos_t = nullptr;   // [ctx][hd/2]
    const float* sin_t = nullptr;
    float eps = 0.f;
    float* k_cache = nullptr;       // [kv][ctx][hd]
    float* v_cache = nullptr;
    const int32_t* pos = nullptr;
    int heads = 0, kv = 0, hd = 0, ctx = 0;
    float* out = nullptr;           // [heads][hd]
    int8_t* outq = nullptr;         // optional quantized output
    int8_t* outl = nullptr;         // with outq: the two-word form's low words
    float* outs = nullptr;
    int* err = nullptr;             // bit 2 set for a position outside [0, ctx)
    // batch form: `batch` sequences, sequence b's rows at b * (heads or kv) * hd, caches at b * cache_stride, position
    // pos[b], outputs at b * heads * hd
    int batch = 1;
    int64_t cache_stride = 0;
    L2Prefetch pf;                       // weights of later launches to fetch into L2 at the start
    int pdl = 0;
};
void attention_scratch(const AttnCall& c, size_t* bytes, size_t* counters);
cudaError_t launch_attention(const AttnCall& c, Carve& ws, cudaStream_t st);

struct ArgmaxCall {
    const float* x = nullptr;
    int64_t n = 0;
    int32_t* tok = nullptr;     // written with the argmax
    int32_t* pos = nullptr;     // incremented (when not null)
    const int* err = nullptr;   // when set and non-zero, tok and pos are left unchanged
    int ctx = 0;                // with pos: a position outside [0, ctx) leaves tok and pos unchanged
    int rows = 1;               // a batch: rows of n logits (row r at x + r * n), each with its own tok[r] and pos[r]
    L2Prefetch pf;                       // weights of later launches to fetch into L2 at the start
    int pdl = 0;
};
void argmax_scratch(const ArgmaxCall& c, size_t* bytes, size_t* counters);
cudaError_t launch_argmax(const ArgmaxCall& c, Carve& ws, cudaStream_t st);

cudaError_t launch_rope_table(float* cos_t, float* sin_t, int ctx, int half, double theta, cudaStream_t st);

// A chunk of token rows: the residual rows gathered from the embedding and each row's position (*pos + r).
cudaError_t launch_chunk_setup(const int32_t* tokens, int64_t rows, const float* embed, int64_t D, int64_t vocab,
                               const int32_t* pos, int ctx, int32_t* posr, float* h, int* err, cudaStream_t st);
// Causal attention of a chunk of rows (row r at position posr[r]): QK-norm + RoPE of every row and the cache append
// first, then the rows attend their positions, split over position groups and folded.
struct ChunkAttnCall {
    const float* q = nullptr;       // [rows][heads][hd], before QK-norm and RoPE
    const float* k = nullptr;       // [rows][kv][hd]
    const float* v = nullptr;       // [rows][kv][hd]
    const float* q_norm = nullptr;
    const float* k_norm = nullptr;
    const float* cos_t = nullptr;
    const float* sin_t = nullptr;
    float eps = 0.f;
    float* k_cache = nullptr;       // [kv][ctx][hd]
    float* v_cache = nullptr;
    const int32_t* posr = nullptr;  // [rows]
    int64_t rows = 0;
    int heads = 0, kv = 0, hd = 0, ctx = 0;
    float* out = nullptr;           // [rows][heads][hd]
    int8_t* outq = nullptr;         // optional quantized output
    int8_t* outl = nullptr;         // with outq: the two-word form's low words
    float* outs = nullptr;
    int* err = nullptr;             // error word: bit 8 when the tensor-core form meets a value that is not finite
};
void chunk_attention_scratch(int64_t rows, int heads, int ctx, size_t* bytes);
cudaError_t launch_chunk_attention(const ChunkAttnCall& c, Carve& ws, cudaStream_t st);

// *pos += add on the device, unless *err is set.
cudaError_t launch_pos_add(int32_t* pos, int add, const int* err, cudaStream_t st);

// The scratch and counters of a caller's workspace, for the launches of one call (the C ABI's q8_ws).
Carve workspace_carve(const q8_ws* ws);

// A persistent grid for `kernel`: enough CTAs of Q8_THREADS threads for `warps` warps, at most the CTAs that fit on
// the device at once (occupancy times SMs).
// ---- the decode step's layers in one persistent launch (decode_persistent.cu) ----------------------------------
// One layer's matrices and vectors, as the persistent kernel reads them (a device array of these, one per layer).
struct PersistLayer {
    const int8_t *wq_q, *wk_q, *wv_q, *wo_q, *wr_q, *wg_q, *wu_q, *wd_q;  // quants
    const float *wq_s, *wk_s, *wv_s, *wo_s, *wr_s, *wg_s, *wu_s, *wd_s;   // block scales
    const float *attn_norm, *ffn_norm, *q_norm, *k_norm;
    float *kc, *vc;  // this layer's caches [kv][ctx][hd]
};

// The shapes the kernel is sized for, and how it deals each phase's work to the CTAs (one CTA per SM).
struct PersistDims {
    int L = 0, D = 0, H = 0, KV = 0, E = 0, K = 0, F = 0, ctx = 0, mode = 0;
};
// Byte offsets in a CTA's shared memory (computed on the host; the kernel reads them from its parameters).
struct PersistLayout {
    uint32_t xq = 0, xl = 0, xs = 0;     // the normed activation's words (and low words) and scales
    uint32_t u = 0;                      // per-stage scratch (a union over the stages)
    uint32_t w = 0, c = 0, r = 0;        // the weight regions
    uint32_t total = 0;
    // inside u
    uint32_t b_qs = 0, b_kn = 0, b_vn = 0, b_sc = 0, b_red = 0;  // attention
    uint32_t f_red = 0;                                        // fold: the warps' sums
    uint32_t o_q = 0, o_l = 0, o_s = 0;                        // O: the attention output's words and scales
    uint32_t e_key = 0, e_val = 0;                             // routing
    uint32_t d_q = 0, d_l = 0, d_s = 0;                        // down: the hidden rows' words and scales
    uint32_t red_in_c = 0;  // the attention's value sums meet at b_red in the C region (else in u)
};
struct PersistPlan {
    int ok = 0;          // 0: the shapes do not fit the kernel (why: in `why`)
    const char* why = "";
    int nb = 0;          // CTAs (one per SM)
    int rq = 0, ro = 0, rr = 0, rd = 0;  // q/k/v, O, router and down rows per CTA
    int ppg = 0;         // attention CTAs per key/value head
    int capr = 0;        // cache positions a CTA stages (its share at the longest cache)
    int gu = 0;          // gate-up items (row pairs) per CTA
    size_t smem = 0;     // dynamic shared memory per CTA
    PersistLayout lay;
};
PersistPlan persist_plan(const PersistDims& d);

struct PersistCall {
    PersistDims dims;
    PersistPlan plan;
    const PersistLayer* layers = nullptr;  // device [L]
    float eps = 0.f, scale = 0.f;
    const float* embed = nullptr;
    int64_t vocab = 0;
    const int32_t* tok = nullptr;
    const int32_t* pos = nullptr;
    const float *cos_t = nullptr, *sin_t = nullptr;
    float *h = nullptr, *q = nullptr, *k = nullptr, *v = nullptr;
    float* part = nullptr;                 // [H][ppg][hd + 2] attention partials
    float* att = nullptr;
    int8_t *attq = nullptr, *attl = nullptr;
    float* atts = nullptr;
    float* logits = nullptr;               // [E]
    int32_t* ids = nullptr;
    float* gates = nullptr;
    float* hbuf = nullptr;                 // [K * F]
    int8_t *hq = nullptr, *hl = nullptr;   // the hidden rows' words (and low words) [K * F] and scales [K * F / 32]
    float* hs = nullptr;
    int* qcnt = nullptr;                   // [K * F / 32] arrivals per 32-row block (left zero)
    float* trace = nullptr;                // optional [L + 1][D]
    unsigned* bar = nullptr;               // kPersistBarBytes: grid-barrier arrival and exit counters, zero between
                                           // launches
    int* err = nullptr;
};
cudaError_t launch_persist(const PersistCall& c, cudaStream_t st);
constexpr size_t kPersistBarBytes = 2048;  // the grid barrier's counters, each on a 128-byte line of its own
extern int kPersistentDecode;  // q8_set_persistent_decode

template <typename Kern>
int persistent_grid(Kern kernel, size_t smem, int64_t warps) {
    int occ = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, 256, smem) != cudaSuccess || occ < 1) occ = 1;
    int64_t ctas = (warps + 7) / 8;
    const int64_t cap = (int64_t)device_info().sms * occ;
    if (ctas > cap) ctas = cap;
    if (ctas < 1) ctas = 1;
    return (int)ctas;
}

// Launch helper: programmatic dependent launch when requested.
template <typename Kern, typename... Args>
cudaError_t launch(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, int pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace q8
