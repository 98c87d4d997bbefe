// The decode step of a whole model: its launches in order and the CUDA graph they are captured into.
//
// What it computes: qwen_emit docs, emit_qwen30b_generate (RMSNorm -> Q/K/V -> per-head QK-norm + RoPE -> attention
// over the KV cache -> O-proj -> residual -> RMSNorm -> 8-of-128 mixture -> residual per layer; the LM head; a T=1
// step captured as one CUDA graph and replayed per token with position and token on the device) and forward_shim.rs
// (module docs: the whole forward captured as one CUDA graph; every stage reads and writes whole buffers).
//
// Launches per layer (the merges are GB300 choices, not the pages'): one projection for q, k and v together that first
// forms RMSNorm of the residual row itself (the first layer gathers the token's embedding row into the residual
// stream); one split attention that first applies QK-norm and RoPE and appends the new key and value rows (its fold
// quantizes the result for the O projection); the O projection with the residual sum in its epilogue; the router
// projection with its RMSNorm and its top-k in one cluster launch; gate-up; down-and-combine with the residual sum in
// its epilogue.  Then the LM head with the final norm, and the arg-max that advances token and position.  Shapes the
// fused forms do not take fall back to a separate add+RMSNorm launch.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <vector>

#include "kernels.h"
#include "q8moe.h"
#include "stream.cuh"

namespace q8 {
extern int model_fail(int code, const char* fmt, ...);
}

using namespace q8;

struct q8_model {
    q8_model_desc d;
    std::vector<const float*> attn_norm, ffn_norm, q_norm, k_norm;
    std::vector<q8_mat> wq, wk, wv, wo, router, gate, up, down;
    std::vector<q8_mat> sgate, sup, sdown;  // the shared expert per layer (empty when there is none)
    std::vector<const float*> router_f32;   // f32 routers per layer (empty when the routers are Q8_0)
    std::vector<float*> kc, vc;
    char* arena = nullptr;
    size_t arena_bytes = 0;
    float *h = nullptr, *x = nullptr, *q = nullptr, *k = nullptr, *v = nullptr, *att = nullptr, *logits = nullptr;
    float *cos_t = nullptr, *sin_t = nullptr, *hbuf = nullptr, *gates = nullptr, *rlog = nullptr;
    int8_t *xq = nullptr, *attq = nullptr, *hq = nullptr;
    int8_t *xl = nullptr, *attl = nullptr, *hl = nullptr;  // the two-word mode's low words
    float *xs = nullptr, *atts = nullptr, *hs = nullptr;
    int32_t* ids = nullptr;
    PlanPtrs plan;                 // batch form: the sequences' choices grouped by expert
    int64_t B = 1;                 // sequences per step
    int* err = nullptr;
    char* ws = nullptr;
    size_t ws_bytes = 0;
    int* counters = nullptr;
    size_t n_counters = 0;
    cudaStream_t cap = nullptr;
    cudaGraphExec_t exec = nullptr;
    int64_t kernels_per_step = 0;  // kernel nodes of the captured step
    int pdl = 1;       // programmatic dependent launch between the step's kernels
    // the step's layers as one persistent launch (when the shapes fit it): its plan, layer table, attention partials
    // and grid-barrier counters, in one allocation
    PersistPlan pplan;
    char* pstate = nullptr;
    PersistLayer* players = nullptr;
    float* ppart = nullptr;
    unsigned* pbar = nullptr;
    int* pqcnt = nullptr;
};

namespace {

int check_mat_shape(const q8_mat& m, int64_t rows, int64_t cols, const char* name, int64_t layer) {
    if (!m.q || !m.s) return model_fail(Q8_EINVAL, "%s[%lld]: null quants or scales", name, (long long)layer);
    if (m.rows != rows || m.cols != cols)
        return model_fail(Q8_EINVAL, "%s[%lld]: %lld x %lld, expected %lld x %lld", name, (long long)layer,
                          (long long)m.rows, (long long)m.cols, (long long)rows, (long long)cols);
    if ((uintptr_t)m.q % 32) return model_fail(Q8_EINVAL, "%s[%lld]: quants not 32-byte aligned", name, (long long)layer);
    if ((uintptr_t)m.s % 4) return model_fail(Q8_EINVAL, "%s[%lld]: scales not 4-byte aligned", name, (long long)layer);
    return Q8_OK;
}

template <typename T>
T* carve_arena(char*& at, size_t n) {
    uintptr_t p = ((uintptr_t)at + 255) & ~uintptr_t(255);
    at = (char*)(p + n * sizeof(T));
    return (T*)p;
}

Carve fresh_carve(q8_model* m) {
    Carve c;
    c.base = m->ws;
    c.size = m->ws_bytes;
    c.counters = m->counters;
    c.n_counters = m->n_counters;
    return c;
}

// The step's launches in order.  With `trace` (device f32 [layers + 1][d]) the residual stream entering the first layer
// (the token's embedding row) and leaving each layer is copied out after the launch that completes it (a debug export;
// the copies are ordinary stream operations between the kernels).
cudaError_t step_launches(q8_model* m, cudaStream_t st, float* trace = nullptr) {
    const q8_model_desc& d = m->d;
    const int mode = (int)d.mode;
    const int64_t D = d.d, H = d.heads, KV = d.kv_heads, HD = d.head_dim;
    const int pdl = m->pdl;
    cudaError_t e = cudaSuccess;
#define Q8_TRY(x)                    \
    do {                             \
        e = (x);                     \
        if (e != cudaSuccess) return e; \
    } while (0)
    const bool persistent = kPersistentDecode && m->pplan.ok;
    if (persistent) {
        PersistCall c;
        c.dims.L = (int)d.layers;
        c.dims.D = (int)D;
        c.dims.H = (int)H;
        c.dims.KV = (int)KV;
        c.dims.E = (int)d.experts;
        c.dims.K = (int)d.k;
        c.dims.F = (int)d.dff;
        c.dims.ctx = (int)d.ctx;
        c.dims.mode = mode;
        c.plan = m->pplan;
        c.layers = m->players;
        c.eps = d.eps;
        c.scale = (float)(1.0 / sqrt((double)HD));
        c.embed = d.embed;
        c.vocab = d.vocab;
        c.tok = d.tok;
        c.pos = d.pos;
        c.cos_t = m->cos_t;
        c.sin_t = m->sin_t;
        c.h = m->h;
        c.q = m->q;
        c.k = m->k;
        c.v = m->v;
        c.part = m->ppart;
        c.att = m->att;
        c.attq = m->attq;
        c.attl = m->attl;
        c.atts = m->atts;
        c.logits = m->rlog;
        c.ids = m->ids;
        c.gates = m->gates;
        c.hbuf = m->hbuf;
        c.hq = m->hq;
        c.hl = m->hl;
        c.hs = m->hs;
        c.qcnt = m->pqcnt;
        c.trace = trace;
        c.bar = m->pbar;
        c.err = m->err;
        Q8_TRY(launch_persist(c, st));
    }
    for (int64_t l = 0; !persistent && l < d.layers; ++l) {
        // attention half: norm (the first layer gathers the token's embedding row into the residual stream), then q,
        // k and v in one projection launch; the norm runs inside the projection launch when the shapes allow it
        GemvCall g;
        g.mode = mode;
        g.k = D;
        g.nseg = 3;
        g.seg[0] = GemvSeg{m->wq[l].q, m->wq[l].s, H * HD, m->q, nullptr};
        g.seg[1] = GemvSeg{m->wk[l].q, m->wk[l].s, KV * HD, m->k, nullptr};
        g.seg[2] = GemvSeg{m->wv[l].q, m->wv[l].s, KV * HD, m->v, nullptr};
        g.x = m->x;
        g.xq = m->xq;
        g.xl = m->xl;
        g.xs = m->xs;
        g.pdl = pdl;
        g.err = m->err;
        g.norm_a = l == 0 ? d.embed : m->h;
        g.norm_a_row = l == 0 ? d.tok : nullptr;
        g.norm_a_rows = d.vocab;
        g.norm_w = m->attn_norm[l];
        g.eps = d.eps;
        g.norm_sum_out = l == 0 ? m->h : nullptr;
        if (!gemv_norm_supported(g)) {
            g.norm_a = nullptr;
            g.norm_a_row = nullptr;
            g.norm_sum_out = nullptr;
            NormCall n;
            if (l == 0) {
                n.a = d.embed;
                n.a_row = d.tok;
                n.a_rows = d.vocab;
                n.sum = m->h;
            } else {
                n.a = m->h;
            }
            n.w = m->attn_norm[l];
            n.rows = 1;
            n.d = D;
            n.eps = d.eps;
            if (mode == 0) n.y = m->x;
            else {
                n.yq = m->xq;
                n.yl = m->xl;
                n.ys = m->xs;
            }
            n.err = m->err;
            n.pdl = pdl;
            Q8_TRY(launch_add_rmsnorm(n, st));
        }
        {
            Carve cv = fresh_carve(m);
            Q8_TRY(launch_gemv(g, cv, st));
        }
        if (trace && l == 0)
            Q8_TRY(cudaMemcpyAsync(trace, m->h, (size_t)D * sizeof(float), cudaMemcpyDeviceToDevice, st));
        {
            Carve cv = fresh_carve(m);
            AttnCall a;  // QK-norm, RoPE and the cache append happen inside the attention launch
            a.q = m->q;
            a.k = m->k;
            a.v = m->v;
            a.q_norm = m->q_norm[l];
            a.k_norm = m->k_norm[l];
            a.cos_t = m->cos_t;
            a.sin_t = m->sin_t;
            a.eps = d.eps;
            a.err = m->err;
            a.k_cache = m->kc[l];
            a.v_cache = m->vc[l];
            a.pos = d.pos;
            a.heads = (int)H;
            a.kv = (int)KV;
            a.hd = (int)HD;
            a.ctx = (int)d.ctx;
            a.out = m->att;
            if (mode >= 1) {
                a.outq = m->attq;
                a.outl = m->attl;
                a.outs = m->atts;
            }
            a.pdl = pdl;
            Q8_TRY(launch_attention(a, cv, st));
        }
        {
            Carve cv = fresh_carve(m);
            GemvCall g;
            g.mode = mode;
            g.k = H * HD;
            g.seg[0] = GemvSeg{m->wo[l].q, m->wo[l].s, D, m->h, m->h};  // h = h + o
            g.x = m->att;
            g.xq = m->attq;
            g.xl = m->attl;
            g.xs = m->atts;
            g.pdl = pdl;
            g.err = m->err;
            Q8_TRY(launch_gemv(g, cv, st));
        }
        // feed-forward half: the norm happens inside the router launch when the shapes allow it (a router of f32
        // values reads the f32 activation: a norm launch writes it, and the int8 form the experts read)
        const bool rf = !m->router_f32.empty();
        const bool fused_norm2 =
            !rf && route_row_supported(mode, d.experts, D, (int)d.k) && D % 256 == 0 && D <= 4096;
        if (!fused_norm2) {
            NormCall n2;
            n2.a = m->h;
            n2.w = m->ffn_norm[l];
            n2.rows = 1;
            n2.d = D;
            n2.eps = d.eps;
            if (mode == 0 || rf) n2.y = m->x;
            if (mode != 0) {
                n2.yq = m->xq;
                n2.yl = m->xl;
                n2.ys = m->xs;
            }
            n2.pdl = pdl;
            Q8_TRY(launch_add_rmsnorm(n2, st));
        }
        if (rf) {  // the f32 router's projection, then its top-k
            Q8_TRY(launch_router_f32(m->router_f32[l], d.experts, D, m->x, 1, m->rlog, pdl, st));
            TopkCall t;
            t.logits = m->rlog;
            t.R = 1;
            t.E = d.experts;
            t.K = (int)d.k;
            t.ids = m->ids;
            t.gates = m->gates;
            t.pdl = pdl;
            Q8_TRY(launch_topk(t, st));
        } else if (route_row_supported(mode, d.experts, D, (int)d.k)) {
            // the router projection and its top-k in one cluster launch
            RouteRowCall r;
            r.mode = mode;
            r.q = m->router[l].q;
            r.s = m->router[l].s;
            r.E = d.experts;
            r.d = D;
            r.K = (int)d.k;
            r.x = m->x;
            r.xq = m->xq;
            r.xl = m->xl;
            r.xs = m->xs;
            r.ids = m->ids;
            r.gates = m->gates;
            if (fused_norm2) {
                r.norm_a = m->h;
                r.norm_w = m->ffn_norm[l];
                r.eps = d.eps;
                r.x_out = mode == 0 ? m->x : nullptr;
                r.xq_out = m->xq;
                r.xl_out = m->xl;
                r.xs_out = m->xs;
            }
            r.pdl = pdl;
            Q8_TRY(launch_route_row(r, st));
        } else {
            Carve cv = fresh_carve(m);
            GemvCall g;
            g.mode = mode;
            g.k = D;
            g.seg[0] = GemvSeg{m->router[l].q, m->router[l].s, d.experts, m->rlog, nullptr};
            g.x = m->x;
            g.xq = m->xq;
            g.xl = m->xl;
            g.xs = m->xs;
            g.pdl = pdl;
            g.err = m->err;
            Q8_TRY(launch_gemv(g, cv, st));
            TopkCall t;
            t.logits = m->rlog;
            t.R = 1;
            t.E = d.experts;
            t.K = (int)d.k;
            t.ids = m->ids;
            t.gates = m->gates;
            t.pdl = pdl;
            Q8_TRY(launch_topk(t, st));
        }
        bool hq_by_gate = false;
        {
            Carve cv = fresh_carve(m);
            ExpertCall c;
            c.mode = mode;
            c.q0 = m->gate[l].q;
            c.s0 = m->gate[l].s;
            c.q1 = m->up[l].q;
            c.s1 = m->up[l].s;
            c.E = d.experts;
            c.out_rows = d.dff;
            c.k = D;
            c.R = 1;
            c.K = (int)d.k;
            c.ids = m->ids;
            c.x = m->x;
            c.xq = m->xq;
            c.xl = m->xl;
            c.xs = m->xs;
            c.h = m->hbuf;
            if (!m->sgate.empty()) {  // the shared expert's rows follow the routed ones
                c.sq0 = m->sgate[l].q;
                c.ss0 = m->sgate[l].s;
                c.sq1 = m->sup[l].q;
                c.ss1 = m->sup[l].s;
                c.sdff = d.shared_dff;
            }
            if (mode >= 1 && gate_row_supported(c)) {  // the hidden rows quantized once, by the kernel that forms them
                c.hq_out = m->hq;
                c.hl_out = m->hl;
                c.hs_out = m->hs;
                hq_by_gate = true;
            }
            c.pdl = pdl;
            c.err = m->err;
            Q8_TRY(launch_gate_up(c, cv, st));
        }
        {
            Carve cv = fresh_carve(m);
            ExpertCall c;
            c.mode = mode;
            c.q0 = m->down[l].q;
            c.s0 = m->down[l].s;
            c.E = d.experts;
            c.out_rows = D;
            c.k = d.dff;
            c.R = 1;
            c.K = (int)d.k;
            c.ids = m->ids;
            c.gates = m->gates;
            c.x = m->hbuf;  // f32 hidden rows
            if (hq_by_gate) {  // and their int8 form, written by gate-up
                c.xq = m->hq;
                c.xl = m->hl;
                c.xs = m->hs;
            }
            if (!m->sdown.empty()) {
                c.sq0 = m->sdown[l].q;
                c.ss0 = m->sdown[l].s;
                c.sdff = d.shared_dff;
            }
            c.residual = m->h;  // h = h + mixture
            c.y = m->h;
            c.pdl = pdl;
            c.err = m->err;
            Q8_TRY(launch_down_combine(c, cv, st));
        }
        if (trace)
            Q8_TRY(cudaMemcpyAsync(trace + (l + 1) * D, m->h, (size_t)D * sizeof(float), cudaMemcpyDeviceToDevice,
                                   st));
    }
    // final norm (inside the LM head launch when the shapes allow it), LM head, greedy token
    {
        GemvCall g;
        g.mode = mode;
        g.k = D;
        g.seg[0] = GemvSeg{d.lm_head.q, d.lm_head.s, d.vocab, m->logits, nullptr};
        g.x = m->x;
        g.xq = m->xq;
        g.xl = m->xl;
        g.xs = m->xs;
        // after the persistent launch the LM head waits for it to end: programmatic dependent launch is not relied on
        // behind a cooperative launch (logits read part of a residual row the layers were still writing)
        g.pdl = persistent ? 0 : pdl;
        g.err = m->err;
        g.norm_a = m->h;
        g.norm_w = d.final_norm;
        g.eps = d.eps;
        if (!gemv_norm_supported(g)) {
            g.norm_a = nullptr;
            NormCall nf;
            nf.a = m->h;
            nf.w = d.final_norm;
            nf.rows = 1;
            nf.d = D;
            nf.eps = d.eps;
            if (mode == 0) nf.y = m->x;
            else {
                nf.yq = m->xq;
                nf.yl = m->xl;
                nf.ys = m->xs;
            }
            nf.pdl = pdl;
            Q8_TRY(launch_add_rmsnorm(nf, st));
        }
        Carve cv = fresh_carve(m);
        Q8_TRY(launch_gemv(g, cv, st));
    }
    {
        Carve cv = fresh_carve(m);
        ArgmaxCall a;
        a.x = m->logits;
        a.n = d.vocab;
        a.tok = d.tok;
        a.pos = d.pos;
        a.err = m->err;
        a.ctx = (int)d.ctx;
        a.pdl = pdl;
        Q8_TRY(launch_argmax(a, cv, st));
    }
#undef Q8_TRY
    return cudaSuccess;
}

// The batch form's step (lane/mod.rs: FormKind::Batch): the sequences are the rows of one chunk for every norm,
// projection and the mixture (each weight read once for all of them, each chosen expert once for the sequences that
// chose it), and each attends its own cache at its own position.  Plain launches in order.
cudaError_t batch_step_launches(q8_model* m, cudaStream_t st, float* trace = nullptr) {
    const q8_model_desc& d = m->d;
    const int mode = (int)d.mode;
    const int64_t B = m->B, D = d.d, H = d.heads, KV = d.kv_heads, HD = d.head_dim, E = d.experts, K = d.k, F = d.dff;
    const bool rf = !m->router_f32.empty();
    const int64_t SF = m->sgate.empty() ? 0 : d.shared_dff;
    cudaError_t e = cudaSuccess;
#define Q8_TRY(x)                       \
    do {                                \
        e = (x);                        \
        if (e != cudaSuccess) return e; \
    } while (0)
    auto norm = [&](const float* a, const int32_t* a_row, const float* w, float* sum) {
        NormCall n;
        n.a = a;
        n.a_row = a_row;
        n.a_rows = d.vocab;
        n.w = w;
        n.rows = B;
        n.d = D;
        n.eps = d.eps;
        n.sum = sum;
        if (mode == 0 || rf) n.y = m->x;
        if (mode != 0) {
            n.yq = m->xq;
            n.yl = m->xl;
            n.ys = m->xs;
        }
        n.err = m->err;
        n.pdl = m->pdl;
        return launch_add_rmsnorm(n, st);
    };
    for (int64_t l = 0; l < d.layers; ++l) {
        // the first layer gathers each sequence's embedding row into its residual row
        Q8_TRY(norm(l == 0 ? d.embed : m->h, l == 0 ? d.tok : nullptr, m->attn_norm[l], l == 0 ? m->h : nullptr));
        if (trace && l == 0)
            Q8_TRY(cudaMemcpyAsync(trace, m->h, (size_t)(B * D) * sizeof(float), cudaMemcpyDeviceToDevice, st));
        {
            GemvCall g;
            g.mode = mode;
            g.k = D;
            g.R = B;
            g.nseg = 3;
            g.seg[0] = GemvSeg{m->wq[l].q, m->wq[l].s, H * HD, m->q, nullptr};
            g.seg[1] = GemvSeg{m->wk[l].q, m->wk[l].s, KV * HD, m->k, nullptr};
            g.seg[2] = GemvSeg{m->wv[l].q, m->wv[l].s, KV * HD, m->v, nullptr};
            g.x = m->x;
            g.xq = m->xq;
            g.xl = m->xl;
            g.xs = m->xs;
            g.err = m->err;
            g.pdl = m->pdl;
            Carve cv = fresh_carve(m);
            Q8_TRY(launch_gemv(g, cv, st));
        }
        {
            AttnCall a;
            a.q = m->q;
            a.k = m->k;
            a.v = m->v;
            a.q_norm = m->q_norm[l];
            a.k_norm = m->k_norm[l];
            a.cos_t = m->cos_t;
            a.sin_t = m->sin_t;
            a.eps = d.eps;
            a.err = m->err;
            a.k_cache = m->kc[l];
            a.v_cache = m->vc[l];
            a.pos = d.pos;
            a.heads = (int)H;
            a.kv = (int)KV;
            a.hd = (int)HD;
            a.ctx = (int)d.ctx;
            a.out = m->att;
            if (mode >= 1) {
                a.outq = m->attq;
                a.outl = m->attl;
                a.outs = m->atts;
            }
            a.batch = (int)B;
            a.cache_stride = KV * d.ctx * HD;
            a.pdl = m->pdl;
            Carve cv = fresh_carve(m);
            Q8_TRY(launch_attention(a, cv, st));
        }
        {
            GemvCall g;
            g.mode = mode;
            g.k = H * HD;
            g.R = B;
            g.seg[0] = GemvSeg{m->wo[l].q, m->wo[l].s, D, m->h, m->h};  // h = h + o
            g.x = m->att;
            g.xq = m->attq;
            g.xl = m->attl;
            g.xs = m->atts;
            g.err = m->err;
            g.pdl = m->pdl;
            Carve cv = fresh_carve(m);
            Q8_TRY(launch_gemv(g, cv, st));
        }
        Q8_TRY(norm(m->h, nullptr, m->ffn_norm[l], nullptr));
        if (rf) {
            Q8_TRY(launch_router_f32(m->router_f32[l], E, D, m->x, B, m->rlog, 0, st));
        } else {
            GemvCall g;
            g.mode = mode;
            g.k = D;
            g.R = B;
            g.seg[0] = GemvSeg{m->router[l].q, m->router[l].s, E, m->rlog, nullptr};
            g.x = m->x;
            g.xq = m->xq;
            g.xl = m->xl;
            g.xs = m->xs;
            g.err = m->err;
            g.pdl = m->pdl;
            Carve cv = fresh_carve(m);
            Q8_TRY(launch_gemv(g, cv, st));
        }
        {
            Carve cv = fresh_carve(m);
            TopkCall t;
            t.logits = m->rlog;
            t.R = B;
            t.E = E;
            t.K = (int)K;
            t.ids = m->ids;
            t.gates = m->gates;
            t.plan = m->plan;
            t.done = cv.take_counters(1);
            t.pdl = m->pdl;
            Q8_TRY(launch_topk(t, st));
        }
        {
            ExpertCall c;
            c.mode = mode;
            c.q0 = m->gate[l].q;
            c.s0 = m->gate[l].s;
            c.q1 = m->up[l].q;
            c.s1 = m->up[l].s;
            c.E = E;
            c.out_rows = F;
            c.k = D;
            c.R = B;
            c.K = (int)K;
            c.ids = m->ids;
            c.x = m->x;
            c.xq = m->xq;
            c.xl = m->xl;
            c.xs = m->xs;
            c.h = m->hbuf;
            c.plan = m->plan;
            c.err = m->err;
            c.pdl = m->pdl;
            if (SF) {
                c.sq0 = m->sgate[l].q;
                c.ss0 = m->sgate[l].s;
                c.sq1 = m->sup[l].q;
                c.ss1 = m->sup[l].s;
                c.sdff = SF;
            }
            Carve cv = fresh_carve(m);
            Q8_TRY(launch_gate_up(c, cv, st));
            if (mode >= 1) Q8_TRY(launch_quantize(m->hbuf, B * (K * F + SF), m->hq, m->hs, st, m->hl));
        }
        {
            ExpertCall c;
            c.mode = mode;
            c.q0 = m->down[l].q;
            c.s0 = m->down[l].s;
            c.E = E;
            c.out_rows = D;
            c.k = F;
            c.R = B;
            c.K = (int)K;
            c.ids = m->ids;
            c.gates = m->gates;
            c.x = mode >= 1 ? nullptr : m->hbuf;
            c.xq = m->hq;
            c.xl = m->hl;
            c.xs = m->hs;
            c.plan = m->plan;
            c.err = m->err;
            c.pdl = m->pdl;
            if (SF) {
                c.sq0 = m->sdown[l].q;
                c.ss0 = m->sdown[l].s;
                c.sdff = SF;
            }
            c.residual = m->h;  // h = h + mixture
            c.y = m->h;
            Carve cv = fresh_carve(m);
            Q8_TRY(launch_down_combine(c, cv, st));
        }
        if (trace)
            Q8_TRY(cudaMemcpyAsync(trace + (l + 1) * B * D, m->h, (size_t)(B * D) * sizeof(float),
                                   cudaMemcpyDeviceToDevice, st));
    }
    // each sequence's final norm, LM head row and greedy token
    Q8_TRY(norm(m->h, nullptr, d.final_norm, nullptr));
    {
        GemvCall g;
        g.mode = mode;
        g.k = D;
        g.R = B;
        g.seg[0] = GemvSeg{d.lm_head.q, d.lm_head.s, d.vocab, m->logits, nullptr};
        g.x = m->x;
        g.xq = m->xq;
        g.xl = m->xl;
        g.xs = m->xs;
        g.err = m->err;
        g.pdl = m->pdl;
        Carve cv = fresh_carve(m);
        Q8_TRY(launch_gemv(g, cv, st));
    }
    {  // every sequence's arg-max in one launch (a row of CTAs per sequence)
        ArgmaxCall a;
        a.x = m->logits;
        a.n = d.vocab;
        a.tok = d.tok;
        a.pos = d.pos;
        a.err = m->err;
        a.ctx = (int)d.ctx;
        a.rows = (int)B;
        a.pdl = m->pdl;
        Carve cv = fresh_carve(m);
        Q8_TRY(launch_argmax(a, cv, st));
    }
#undef Q8_TRY
    return cudaSuccess;
}

// A wait that is bound to give up: one thread waits on a barrier that nothing arrives on, at most `polls` polls, and
// records the timeout in the error word as every pipeline wait of the step does.
__global__ void wait_selftest_kernel(int* err, unsigned polls) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_wait(&bar, 0, err, polls);
}

}  // namespace

extern "C" {

int q8_model_wait_selftest(q8_model* m, unsigned polls, q8_stream stream) {
    if (!m) return model_fail(Q8_EINVAL, "model: null");
    if (polls < 1 || polls > (1u << 20)) return model_fail(Q8_EINVAL, "polls %u: 1 to 2^20", polls);
    wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(m->err, polls);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? Q8_OK : model_fail(Q8_ECUDA, "q8_model_wait_selftest: %s", cudaGetErrorString(e));
}

int q8_model_create(const q8_model_desc* desc, q8_model** out) {
    if (!out) return model_fail(Q8_EINVAL, "model: null");
    *out = nullptr;
    if (!desc) return model_fail(Q8_EINVAL, "desc: null");
    const q8_model_desc& d = *desc;
    if (d.mode != Q8_F32ACT_F64SUM && d.mode != Q8_INT8ACT && d.mode != Q8_INT8ACT2)
        return model_fail(Q8_EINVAL, "mode %d", (int)d.mode);
    if (d.layers < 1 || d.d < 32 || d.heads < 1 || d.kv_heads < 1 || d.vocab < 1 || d.ctx < 1 || d.experts < 1 ||
        d.dff < 32)
        return model_fail(Q8_EINVAL, "a size below its minimum (layers, d, heads, kv_heads, vocab, ctx, experts, dff)");
    if (d.head_dim != 128) return model_fail(Q8_EUNSUPPORTED, "head_dim %lld: the attention kernel is built for 128",
                                             (long long)d.head_dim);
    if (d.heads % d.kv_heads) return model_fail(Q8_EUNSUPPORTED, "query heads that do not group evenly over the key/value heads");
    if (d.heads / d.kv_heads > 8) return model_fail(Q8_EUNSUPPORTED, "more than 8 query heads per key/value head");
    if (d.d % 32 || d.dff % 32) return model_fail(Q8_EUNSUPPORTED, "d and dff must be whole 32-value blocks");
    if (d.d > 8192) return model_fail(Q8_EUNSUPPORTED, "d %lld: a row kernel holds at most 8192 values", (long long)d.d);
    if (d.k < 1 || d.k > 32 || d.k > d.experts) return model_fail(Q8_EUNSUPPORTED, "k %lld: 1 to 32 kept experts", (long long)d.k);
    if (d.experts > 8192) return model_fail(Q8_EUNSUPPORTED, "%lld experts: at most 8192", (long long)d.experts);
    if (d.ctx > (1 << 24) || d.vocab > (1 << 30)) return model_fail(Q8_EUNSUPPORTED, "ctx or vocab past the index range");
    if (!(d.eps >= 0.f) || !(d.rope_theta > 0.0)) return model_fail(Q8_EINVAL, "eps or rope_theta out of range");
    if (d.batch < 0 || d.batch > 64) return model_fail(Q8_EUNSUPPORTED, "batch %lld: 1 to 64 sequences", (long long)d.batch);
    if (d.batch > 1 && d.batch * d.k > 65536) return model_fail(Q8_EUNSUPPORTED, "batch * k: too many choices");
    if (!d.embed || !d.final_norm || !d.tok || !d.pos) return model_fail(Q8_EINVAL, "embed, final_norm, tok or pos: null");
    if (!d.attn_norm || !d.ffn_norm || !d.q_norm || !d.k_norm || !d.wq || !d.wk || !d.wv || !d.wo || !d.router ||
        !d.gate || !d.up || !d.down || !d.k_cache || !d.v_cache)
        return model_fail(Q8_EINVAL, "a per-layer array: null");
    const int64_t D = d.d, QD = d.heads * d.head_dim, KD = d.kv_heads * d.head_dim;
    for (int64_t l = 0; l < d.layers; ++l) {
        if (!d.attn_norm[l] || !d.ffn_norm[l] || !d.q_norm[l] || !d.k_norm[l] || !d.k_cache[l] || !d.v_cache[l])
            return model_fail(Q8_EINVAL, "layer %lld: a null norm weight or cache", (long long)l);
        if ((uintptr_t)d.k_cache[l] % 32 || (uintptr_t)d.v_cache[l] % 32)
            return model_fail(Q8_EINVAL, "layer %lld: a cache not 32-byte aligned", (long long)l);
        int r;
        if ((r = check_mat_shape(d.wq[l], QD, D, "wq", l)) || (r = check_mat_shape(d.wk[l], KD, D, "wk", l)) ||
            (r = check_mat_shape(d.wv[l], KD, D, "wv", l)) || (r = check_mat_shape(d.wo[l], D, QD, "wo", l)) ||
            (r = check_mat_shape(d.router[l], d.experts, D, "router", l)) ||
            (r = check_mat_shape(d.gate[l], d.experts * d.dff, D, "gate", l)) ||
            (r = check_mat_shape(d.up[l], d.experts * d.dff, D, "up", l)) ||
            (r = check_mat_shape(d.down[l], d.experts * D, d.dff, "down", l)))
            return r;
    }
    if (int r = check_mat_shape(d.lm_head, d.vocab, D, "lm_head", 0)) return r;
    const bool has_shared = d.shared_gate || d.shared_up || d.shared_down || d.shared_dff;
    if (has_shared) {
        if (!d.shared_gate || !d.shared_up || !d.shared_down || d.shared_dff < 32)
            return model_fail(Q8_EINVAL, "shared expert: all of shared_gate, shared_up, shared_down and shared_dff");
        if (d.shared_dff % 32) return model_fail(Q8_EUNSUPPORTED, "shared_dff %lld: whole 32-value blocks",
                                                 (long long)d.shared_dff);
        for (int64_t l = 0; l < d.layers; ++l) {
            int r;
            if ((r = check_mat_shape(d.shared_gate[l], d.shared_dff, D, "shared_gate", l)) ||
                (r = check_mat_shape(d.shared_up[l], d.shared_dff, D, "shared_up", l)) ||
                (r = check_mat_shape(d.shared_down[l], D, d.shared_dff, "shared_down", l)))
                return r;
        }
    }
    if (d.router_f32)
        for (int64_t l = 0; l < d.layers; ++l)
            if (!d.router_f32[l] || (uintptr_t)d.router_f32[l] % 16)
                return model_fail(Q8_EINVAL, "router_f32[%lld]: null or not 16-byte aligned", (long long)l);

    q8_model* m = new q8_model();
    m->d = d;
    m->attn_norm.assign(d.attn_norm, d.attn_norm + d.layers);
    m->ffn_norm.assign(d.ffn_norm, d.ffn_norm + d.layers);
    m->q_norm.assign(d.q_norm, d.q_norm + d.layers);
    m->k_norm.assign(d.k_norm, d.k_norm + d.layers);
    m->wq.assign(d.wq, d.wq + d.layers);
    m->wk.assign(d.wk, d.wk + d.layers);
    m->wv.assign(d.wv, d.wv + d.layers);
    m->wo.assign(d.wo, d.wo + d.layers);
    m->router.assign(d.router, d.router + d.layers);
    m->gate.assign(d.gate, d.gate + d.layers);
    m->up.assign(d.up, d.up + d.layers);
    m->down.assign(d.down, d.down + d.layers);
    m->kc.assign(d.k_cache, d.k_cache + d.layers);
    m->vc.assign(d.v_cache, d.v_cache + d.layers);
    if (has_shared) {
        m->sgate.assign(d.shared_gate, d.shared_gate + d.layers);
        m->sup.assign(d.shared_up, d.shared_up + d.layers);
        m->sdown.assign(d.shared_down, d.shared_down + d.layers);
    } else {
        m->d.shared_dff = 0;
    }
    if (d.router_f32) m->router_f32.assign(d.router_f32, d.router_f32 + d.layers);
    m->d.router_f32 = nullptr;
    m->d.shared_gate = m->d.shared_up = m->d.shared_down = nullptr;
    // pointers into the caller's arrays are not kept
    m->d.attn_norm = m->d.ffn_norm = m->d.q_norm = m->d.k_norm = nullptr;
    m->d.wq = m->d.wk = m->d.wv = m->d.wo = m->d.router = m->d.gate = m->d.up = m->d.down = nullptr;
    m->d.k_cache = m->d.v_cache = nullptr;

    // one arena for the step's activations, a row each per sequence (sizes rounded to 256 B each); the hidden rows
    // hold the routed experts' rows and then the shared expert's
    const int64_t B = d.batch > 1 ? d.batch : 1;
    const int64_t KF = B * (d.k * d.dff + (has_shared ? d.shared_dff : 0));
    const size_t half = (size_t)d.head_dim / 2;
    size_t need = 0;
    auto add = [&](size_t bytes) { need += (bytes + 255) & ~size_t(255); };
    add(B * D * 4);          // h
    add(B * D * 4);          // x
    add(B * QD * 4);         // q
    add(B * KD * 4);         // k
    add(B * KD * 4);         // v
    add(B * QD * 4);         // att
    add(d.logits ? 0 : B * d.vocab * 4);
    add(d.ctx * half * 4);  // cos
    add(d.ctx * half * 4);  // sin
    add(KF * 4);         // hbuf
    add(B * d.k * 4);        // gates
    add(B * d.experts * 4);  // router logits
    add(B * D);              // xq
    add(B * D / 32 * 4);     // xs
    add(B * QD);             // attq
    add(B * QD / 32 * 4);    // atts
    add(KF);             // hq
    add(KF / 32 * 4);    // hs
    add(B * D);              // xl
    add(B * QD);             // attl
    add(KF);             // hl
    add(B * d.k * 4);        // ids
    add(d.experts * 4 + (d.experts + 1) * 4 * 2 + B * d.k * 4 + 1024);  // the batch form's grouping
    add(256);            // err
    need += 4096;
    cudaError_t e = cudaMalloc(&m->arena, need);
    if (e != cudaSuccess) {
        delete m;
        return model_fail(Q8_ECUDA, "q8_model_create: %s", cudaGetErrorString(e));
    }
    m->arena_bytes = need;
    char* at = m->arena;
    m->B = B;
    m->h = carve_arena<float>(at, B * D);
    m->x = carve_arena<float>(at, B * D);
    m->q = carve_arena<float>(at, B * QD);
    m->k = carve_arena<float>(at, B * KD);
    m->v = carve_arena<float>(at, B * KD);
    m->att = carve_arena<float>(at, B * QD);
    m->logits = d.logits ? d.logits : carve_arena<float>(at, B * d.vocab);
    m->cos_t = carve_arena<float>(at, d.ctx * half);
    m->sin_t = carve_arena<float>(at, d.ctx * half);
    m->hbuf = carve_arena<float>(at, KF);
    m->gates = carve_arena<float>(at, B * d.k);
    m->rlog = carve_arena<float>(at, B * d.experts);
    m->xq = carve_arena<int8_t>(at, B * D);
    m->xs = carve_arena<float>(at, B * D / 32);
    m->attq = carve_arena<int8_t>(at, B * QD);
    m->atts = carve_arena<float>(at, B * QD / 32);
    m->hq = carve_arena<int8_t>(at, KF);
    m->hs = carve_arena<float>(at, KF / 32);
    m->xl = carve_arena<int8_t>(at, B * D);
    m->attl = carve_arena<int8_t>(at, B * QD);
    m->hl = carve_arena<int8_t>(at, KF);
    m->ids = carve_arena<int32_t>(at, B * d.k);
    m->plan.counts = carve_arena<int32_t>(at, d.experts);
    m->plan.offsets = carve_arena<int32_t>(at, d.experts + 1);
    m->plan.lists = carve_arena<int32_t>(at, B * d.k);
    m->plan.active = carve_arena<int32_t>(at, d.experts + 1);
    m->err = carve_arena<int>(at, 64);
    if (d.mode == Q8_F32ACT_F64SUM) {
        m->xq = nullptr;
        m->xs = nullptr;
        m->attq = nullptr;
        m->atts = nullptr;
        m->hq = nullptr;
        m->hs = nullptr;
    }
    if (d.mode != Q8_INT8ACT2) {
        m->xl = nullptr;
        m->attl = nullptr;
        m->hl = nullptr;
    }
    // workspace: the largest single launch's scratch (launches of a step run one after another)
    m->ws_bytes = size_t(64) << 20;
    m->n_counters = size_t(1) << 20;
    e = cudaMalloc(&m->ws, m->ws_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&m->counters, m->n_counters * sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(m->counters, 0, m->n_counters * sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(m->err, 0, 256);
    if (e == cudaSuccess) e = launch_rope_table(m->cos_t, m->sin_t, (int)d.ctx, (int)half, d.rope_theta, 0);
    // the persistent step: one sequence in an int8 mode, Q8_0 routers, no shared expert, block scales on 16-byte
    // boundaries (the kernel bulk-copies whole rows of them), shapes it fits
    bool scales16 = true;
    for (int64_t l = 0; l < d.layers; ++l)
        for (const q8_mat* w : {&m->wq[l], &m->wk[l], &m->wv[l], &m->wo[l], &m->router[l], &m->gate[l], &m->up[l],
                                &m->down[l]})
            scales16 = scales16 && (uintptr_t)w->s % 16 == 0;
    if (e == cudaSuccess && B == 1 && !has_shared && !d.router_f32 && scales16) {
        PersistDims pd;
        pd.L = (int)d.layers;
        pd.D = (int)D;
        pd.H = (int)d.heads;
        pd.KV = (int)d.kv_heads;
        pd.E = (int)d.experts;
        pd.K = (int)d.k;
        pd.F = (int)d.dff;
        pd.ctx = (int)d.ctx;
        pd.mode = (int)d.mode;
        m->pplan = persist_plan(pd);
        if (m->pplan.ok) {
            const size_t lt = ((size_t)d.layers * sizeof(PersistLayer) + 255) & ~size_t(255);
            const size_t pb = ((size_t)d.heads * m->pplan.ppg * (d.head_dim + 2) * 4 + 255) & ~size_t(255);
            const size_t qc = ((size_t)d.k * d.dff / 32 * 4 + 255) & ~size_t(255);
            e = cudaMalloc(&m->pstate, lt + pb + kPersistBarBytes + qc);
            if (e == cudaSuccess) {
                m->players = reinterpret_cast<PersistLayer*>(m->pstate);
                m->ppart = reinterpret_cast<float*>(m->pstate + lt);
                m->pbar = reinterpret_cast<unsigned*>(m->pstate + lt + pb);
                m->pqcnt = reinterpret_cast<int*>(m->pstate + lt + pb + kPersistBarBytes);
                std::vector<PersistLayer> t((size_t)d.layers);
                for (int64_t l = 0; l < d.layers; ++l) {
                    PersistLayer& y = t[(size_t)l];
                    y.wq_q = m->wq[l].q;
                    y.wq_s = m->wq[l].s;
                    y.wk_q = m->wk[l].q;
                    y.wk_s = m->wk[l].s;
                    y.wv_q = m->wv[l].q;
                    y.wv_s = m->wv[l].s;
                    y.wo_q = m->wo[l].q;
                    y.wo_s = m->wo[l].s;
                    y.wr_q = m->router[l].q;
                    y.wr_s = m->router[l].s;
                    y.wg_q = m->gate[l].q;
                    y.wg_s = m->gate[l].s;
                    y.wu_q = m->up[l].q;
                    y.wu_s = m->up[l].s;
                    y.wd_q = m->down[l].q;
                    y.wd_s = m->down[l].s;
                    y.attn_norm = m->attn_norm[l];
                    y.ffn_norm = m->ffn_norm[l];
                    y.q_norm = m->q_norm[l];
                    y.k_norm = m->k_norm[l];
                    y.kc = m->kc[l];
                    y.vc = m->vc[l];
                }
                e = cudaMemcpy(m->players, t.data(), t.size() * sizeof(PersistLayer), cudaMemcpyHostToDevice);
                if (e == cudaSuccess) e = cudaMemset(m->pbar, 0, kPersistBarBytes + qc);
            }
        }
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        q8_model_destroy(m);
        return model_fail(Q8_ECUDA, "q8_model_create: %s", cudaGetErrorString(e));
    }
    *out = m;
    return Q8_OK;
}

void q8_model_destroy(q8_model* m) {
    if (!m) return;
    if (m->exec) cudaGraphExecDestroy(m->exec);
    if (m->cap) cudaStreamDestroy(m->cap);
    cudaFree(m->arena);
    cudaFree(m->ws);
    cudaFree(m->counters);
    cudaFree(m->pstate);
    delete m;
}

// The step's launches of either form.
static cudaError_t any_step_launches(q8_model* m, cudaStream_t st) {
    return m->B > 1 ? batch_step_launches(m, st) : step_launches(m, st);
}

int decode_step_launches(q8_model* m, q8_stream stream) {
    if (!m) return model_fail(Q8_EINVAL, "model: null");
    cudaError_t e = any_step_launches(m, (cudaStream_t)stream);
    return e == cudaSuccess ? Q8_OK : model_fail(Q8_ECUDA, "decode_step_launches: %s", cudaGetErrorString(e));
}

int decode_step_trace(q8_model* m, float* hidden, q8_stream stream) {
    if (!m) return model_fail(Q8_EINVAL, "model: null");
    if (!hidden || (uintptr_t)hidden % 4) return model_fail(Q8_EINVAL, "hidden: null or misaligned");
    cudaError_t e = m->B > 1 ? batch_step_launches(m, (cudaStream_t)stream, hidden)
                             : step_launches(m, (cudaStream_t)stream, hidden);
    return e == cudaSuccess ? Q8_OK : model_fail(Q8_ECUDA, "decode_step_trace: %s", cudaGetErrorString(e));
}

int decode_step(q8_model* m, q8_stream stream) {
    if (!m) return model_fail(Q8_EINVAL, "model: null");
    cudaError_t e = cudaSuccess;
    if (!m->exec) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing((cudaStream_t)stream, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone)
            return model_fail(Q8_EINVAL, "decode_step: the first call captures the step and cannot run inside a capture");
        if (!m->cap) {
            e = cudaStreamCreateWithFlags(&m->cap, cudaStreamNonBlocking);
            if (e != cudaSuccess) return model_fail(Q8_ECUDA, "decode_step: %s", cudaGetErrorString(e));
        }
        cudaGraph_t graph = nullptr;
        // relaxed: calls other code makes on this thread while the step is captured (a profiler's own synchronizing
        // calls around each launch it intercepts) do not invalidate the capture
        e = cudaStreamBeginCapture(m->cap, cudaStreamCaptureModeRelaxed);
        if (e == cudaSuccess) {
            cudaError_t le = any_step_launches(m, m->cap);
            e = cudaStreamEndCapture(m->cap, &graph);
            if (le != cudaSuccess) e = le;
        }
        if (e == cudaSuccess) {  // the step's kernel count, for callers that report launches
            size_t n = 0;
            e = cudaGraphGetNodes(graph, nullptr, &n);
            std::vector<cudaGraphNode_t> nodes(n);
            if (e == cudaSuccess && n) e = cudaGraphGetNodes(graph, nodes.data(), &n);
            int64_t kernels = 0;
            for (size_t i = 0; e == cudaSuccess && i < n; ++i) {
                cudaGraphNodeType ty;
                e = cudaGraphNodeGetType(nodes[i], &ty);
                if (e == cudaSuccess && ty == cudaGraphNodeTypeKernel) ++kernels;
            }
            m->kernels_per_step = kernels;
        }
        if (e == cudaSuccess) e = cudaGraphInstantiate(&m->exec, graph, 0);
        if (graph) cudaGraphDestroy(graph);
        if (e != cudaSuccess) {
            m->exec = nullptr;
            return model_fail(Q8_ECUDA, "decode_step capture: %s", cudaGetErrorString(e));
        }
    }
    e = cudaGraphLaunch(m->exec, (cudaStream_t)stream);
    return e == cudaSuccess ? Q8_OK : model_fail(Q8_ECUDA, "decode_step: %s", cudaGetErrorString(e));
}

// The prefill launches; with `trace`, the residual rows entering every layer, and the final ones, are copied to
// trace[l][R][d] (l = 0 .. layers).
static int prefill_launches(q8_model* m, const int32_t* tokens, int64_t R, q8_ws* ws, q8_stream stream, float* trace);

int prefill_chunk(q8_model* m, const int32_t* tokens, int64_t R, q8_ws* ws, q8_stream stream) {
    return prefill_launches(m, tokens, R, ws, stream, nullptr);
}

int prefill_chunk_trace(q8_model* m, const int32_t* tokens, int64_t R, q8_ws* ws, float* hidden, q8_stream stream) {
    if (!hidden) return model_fail(Q8_EINVAL, "prefill_chunk_trace: hidden null");
    return prefill_launches(m, tokens, R, ws, stream, hidden);
}

static int prefill_launches(q8_model* m, const int32_t* tokens, int64_t R, q8_ws* ws, q8_stream stream, float* trace) {
    if (!m) return model_fail(Q8_EINVAL, "model: null");
    if (!tokens || !ws) return model_fail(Q8_EINVAL, "prefill_chunk: tokens or ws null");
    if (R < 1 || R > (1 << 20)) return model_fail(Q8_EINVAL, "prefill_chunk: %lld rows", (long long)R);
    if (m->B > 1) return model_fail(Q8_EUNSUPPORTED, "prefill_chunk: one sequence only (the model is a batch form)");
    const q8_model_desc& d = m->d;
    const int mode = (int)d.mode;
    const int64_t D = d.d, H = d.heads, KV = d.kv_heads, HD = d.head_dim, E = d.experts, K = d.k, F = d.dff;
    cudaStream_t st = (cudaStream_t)stream;
    // the chunk's rows, carved from the caller's workspace; every launch's own scratch comes after them
    Carve cb = workspace_carve(ws);
    const bool rf = !m->router_f32.empty();
    const int64_t SF = m->sgate.empty() ? 0 : d.shared_dff;  // the shared expert's hidden width (0: none)
    float* h = cb.take<float>((size_t)(R * D));
    float* x = (mode == 0 || rf) ? cb.take<float>((size_t)(R * D)) : nullptr;  // the f32 router reads f32 rows
    int8_t* xq = mode >= 1 ? cb.take<int8_t>((size_t)(R * D)) : nullptr;
    int8_t* xl = mode == 2 ? cb.take<int8_t>((size_t)(R * D)) : nullptr;
    float* xs = mode >= 1 ? cb.take<float>((size_t)(R * D / 32)) : nullptr;
    float* q = cb.take<float>((size_t)(R * H * HD));
    float* k = cb.take<float>((size_t)(R * KV * HD));
    float* v = cb.take<float>((size_t)(R * KV * HD));
    float* att = cb.take<float>((size_t)(R * H * HD));
    int8_t* attq = mode >= 1 ? cb.take<int8_t>((size_t)(R * H * HD)) : nullptr;
    int8_t* attl = mode == 2 ? cb.take<int8_t>((size_t)(R * H * HD)) : nullptr;
    float* atts = mode >= 1 ? cb.take<float>((size_t)(R * H * HD / 32)) : nullptr;
    float* rlog = cb.take<float>((size_t)(R * E));
    int32_t* ids = cb.take<int32_t>((size_t)(R * K));
    float* gates = cb.take<float>((size_t)(R * K));
    PlanPtrs plan;
    plan.counts = cb.take<int32_t>((size_t)E);
    plan.offsets = cb.take<int32_t>((size_t)E + 1);
    plan.lists = cb.take<int32_t>((size_t)(R * K));
    plan.active = cb.take<int32_t>((size_t)E + 1);
    const int64_t NH = R * K * F + R * SF;  // the routed hidden rows, then the shared expert's
    float* hm = cb.take<float>((size_t)NH);
    int8_t* hmq = mode >= 1 ? cb.take<int8_t>((size_t)NH) : nullptr;
    int8_t* hml = mode == 2 ? cb.take<int8_t>((size_t)NH) : nullptr;
    float* hms = mode >= 1 ? cb.take<float>((size_t)(NH / 32)) : nullptr;
    int32_t* posr = cb.take<int32_t>((size_t)R);
    int* done = cb.take_counters(1);
    if (cb.overflow) return model_fail(Q8_ENOSPACE, "prefill_chunk: workspace too small for %lld rows", (long long)R);
    cudaError_t e = cudaSuccess;
#define Q8_TRY(x)                                                                                                   \
    do {                                                                                                            \
        e = (x);                                                                                                    \
        if (e != cudaSuccess) return model_fail(Q8_ECUDA, "prefill_chunk: %s", cudaGetErrorString(e));             \
    } while (0)
#define Q8_TRY_WS(x, cv)                                                                                            \
    do {                                                                                                            \
        e = (x);                                                                                                    \
        if ((cv).overflow) return model_fail(Q8_ENOSPACE, "prefill_chunk: workspace too small for %lld rows",       \
                                            (long long)R);                                                          \
        if (e != cudaSuccess) return model_fail(Q8_ECUDA, "prefill_chunk: %s", cudaGetErrorString(e));             \
    } while (0)
    auto norm = [&](const float* a, const float* w, int64_t rows) {
        NormCall n;
        n.a = a;
        n.w = w;
        n.rows = rows;
        n.d = D;
        n.eps = d.eps;
        n.y = x;  // f32 rows when the f32 mode or an f32 router reads them
        if (mode != 0) {
            n.yq = xq;
            n.yl = xl;
            n.ys = xs;
        }
        n.err = m->err;
        return launch_add_rmsnorm(n, st);
    };
    // Plain launches in order, no programmatic overlap (each launch reads what the one before it wrote).
    Q8_TRY(launch_chunk_setup(tokens, R, d.embed, D, d.vocab, d.pos, (int)d.ctx, posr, h, m->err, st));
    for (int64_t l = 0; l < d.layers; ++l) {
        if (trace)
            Q8_TRY(cudaMemcpyAsync(trace + l * R * D, h, (size_t)(R * D) * sizeof(float), cudaMemcpyDeviceToDevice, st));
        Q8_TRY(norm(h, m->attn_norm[l], R));
        {
            GemvCall g;
            g.mode = mode;
            g.k = D;
            g.R = R;
            g.nseg = 3;
            g.seg[0] = GemvSeg{m->wq[l].q, m->wq[l].s, H * HD, q, nullptr};
            g.seg[1] = GemvSeg{m->wk[l].q, m->wk[l].s, KV * HD, k, nullptr};
            g.seg[2] = GemvSeg{m->wv[l].q, m->wv[l].s, KV * HD, v, nullptr};
            g.x = x;
            g.xq = xq;
            g.xl = xl;
            g.xs = xs;
            g.err = m->err;
            Carve cv = cb;
            Q8_TRY_WS(launch_gemv(g, cv, st), cv);
        }
        {  // every row's keys and values appended, then each row attends rows 0 .. its position (causal)
            ChunkAttnCall a;
            a.q = q;
            a.k = k;
            a.v = v;
            a.q_norm = m->q_norm[l];
            a.k_norm = m->k_norm[l];
            a.cos_t = m->cos_t;
            a.sin_t = m->sin_t;
            a.eps = d.eps;
            a.k_cache = m->kc[l];
            a.v_cache = m->vc[l];
            a.posr = posr;
            a.rows = R;
            a.heads = (int)H;
            a.kv = (int)KV;
            a.hd = (int)HD;
            a.ctx = (int)d.ctx;
            a.out = att;
            a.outq = attq;
            a.outl = attl;
            a.outs = atts;
            a.err = m->err;
            Carve cv = cb;
            Q8_TRY_WS(launch_chunk_attention(a, cv, st), cv);
        }
        {
            GemvCall g;
            g.mode = mode;
            g.k = H * HD;
            g.R = R;
            g.seg[0] = GemvSeg{m->wo[l].q, m->wo[l].s, D, h, h};  // h = h + o
            g.x = att;
            g.xq = attq;
            g.xl = attl;
            g.xs = atts;
            g.err = m->err;
            Carve cv = cb;
            Q8_TRY_WS(launch_gemv(g, cv, st), cv);
        }
        Q8_TRY(norm(h, m->ffn_norm[l], R));
        {
            if (rf) {
                Q8_TRY(launch_router_f32(m->router_f32[l], E, D, x, R, rlog, 0, st));
            } else {
                GemvCall g;
                g.mode = mode;
                g.k = D;
                g.R = R;
                g.seg[0] = GemvSeg{m->router[l].q, m->router[l].s, E, rlog, nullptr};
                g.x = x;
                g.xq = xq;
                g.xl = xl;
                g.xs = xs;
                g.err = m->err;
                Carve cv = cb;
                Q8_TRY_WS(launch_gemv(g, cv, st), cv);
            }
            TopkCall t;
            t.logits = rlog;
            t.R = R;
            t.E = E;
            t.K = (int)K;
            t.ids = ids;
            t.gates = gates;
            t.plan = plan;
            t.done = done;
            Q8_TRY(launch_topk(t, st));
        }
        {
            ExpertCall c;
            c.mode = mode;
            c.q0 = m->gate[l].q;
            c.s0 = m->gate[l].s;
            c.q1 = m->up[l].q;
            c.s1 = m->up[l].s;
            c.E = E;
            c.out_rows = F;
            c.k = D;
            c.R = R;
            c.K = (int)K;
            c.ids = ids;
            c.x = x;
            c.xq = xq;
            c.xl = xl;
            c.xs = xs;
            c.h = hm;
            c.plan = plan;
            c.err = m->err;
            if (SF) {
                c.sq0 = m->sgate[l].q;
                c.ss0 = m->sgate[l].s;
                c.sq1 = m->sup[l].q;
                c.ss1 = m->sup[l].s;
                c.sdff = SF;
            }
            Carve cv = cb;
            Q8_TRY_WS(launch_gate_up(c, cv, st), cv);
            if (mode >= 1) Q8_TRY(launch_quantize(hm, NH, hmq, hms, st, hml));
        }
        {
            ExpertCall c;
            c.mode = mode;
            c.q0 = m->down[l].q;
            c.s0 = m->down[l].s;
            c.E = E;
            c.out_rows = D;
            c.k = F;
            c.R = R;
            c.K = (int)K;
            c.ids = ids;
            c.gates = gates;
            c.x = mode >= 1 ? nullptr : hm;
            c.xq = hmq;
            c.xl = hml;
            c.xs = hms;
            c.plan = plan;
            c.residual = h;  // h = h + mixture
            c.y = h;
            c.err = m->err;
            if (SF) {
                c.sq0 = m->sdown[l].q;
                c.ss0 = m->sdown[l].s;
                c.sdff = SF;
            }
            Carve cv = cb;
            Q8_TRY_WS(launch_down_combine(c, cv, st), cv);
        }
    }
    if (trace)
        Q8_TRY(cudaMemcpyAsync(trace + d.layers * R * D, h, (size_t)(R * D) * sizeof(float), cudaMemcpyDeviceToDevice,
                               st));
    // the last row's logits and greedy token; the position ends R rows on
    Q8_TRY(launch_pos_add(d.pos, (int)(R - 1), m->err, st));
    {
        NormCall nf;
        nf.a = h + (R - 1) * D;
        nf.w = d.final_norm;
        nf.rows = 1;
        nf.d = D;
        nf.eps = d.eps;
        if (mode == 0) nf.y = m->x;
        else {
            nf.yq = m->xq;
            nf.yl = m->xl;
            nf.ys = m->xs;
        }
        Q8_TRY(launch_add_rmsnorm(nf, st));
        GemvCall g;
        g.mode = mode;
        g.k = D;
        g.seg[0] = GemvSeg{d.lm_head.q, d.lm_head.s, d.vocab, m->logits, nullptr};
        g.x = m->x;
        g.xq = m->xq;
        g.xl = m->xl;
        g.xs = m->xs;
        g.err = m->err;
        Carve cv = cb;
        Q8_TRY_WS(launch_gemv(g, cv, st), cv);
    }
    {
        ArgmaxCall a;
        a.x = m->logits;
        a.n = d.vocab;
        a.tok = d.tok;
        a.pos = d.pos;
        a.err = m->err;
        a.ctx = (int)d.ctx;
        Carve cv = cb;
        Q8_TRY_WS(launch_argmax(a, cv, st), cv);
    }
#undef Q8_TRY
#undef Q8_TRY_WS
    return Q8_OK;
}

int64_t q8_model_launches_per_step(const q8_model* m) { return m ? m->kernels_per_step : 0; }

int q8_model_persistent(const q8_model* m) { return m && kPersistentDecode && m->pplan.ok ? 1 : 0; }

int q8_model_check(q8_model* m, q8_stream stream) {
    if (!m) return model_fail(Q8_EINVAL, "model: null");
    int v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, m->err, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->err, 0, sizeof(int), (cudaStream_t)stream);
    // a persistent step whose wait gave up may have left its grid-barrier counters part-way
    if (e == cudaSuccess && (v & 4) && m->pbar)
        e = cudaMemsetAsync(m->pbar, 0, kPersistBarBytes + ((size_t)m->d.k * m->d.dff / 32 * 4 + 255) / 256 * 256,
                            (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return model_fail(Q8_ECUDA, "q8_model_check: %s", cudaGetErrorString(e));
    if (v & 1) return model_fail(Q8_EINVAL, "a step read a token outside [0, vocab)");
    if (v & 2) return model_fail(Q8_EINVAL, "a step met a position outside [0, ctx)");
    if (v & 4) return model_fail(Q8_ETIMEOUT, "a weight pipeline wait gave up (the step's results are not valid)");
    if (v & 8)
        return model_fail(Q8_EUNSUPPORTED, "a prefill chunk's tensor-core attention met a query, key or value that is "
                                           "not finite");
    return Q8_OK;
}

}  // extern "C"
