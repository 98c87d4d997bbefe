/*
 * CPU oracle — TEST INFRASTRUCTURE ONLY (see oracle.h).  Plain loops, f64 unless the pages fix another precision.
 * Built with -ffp-contract=off and without fast-math, so every f32 operation written here is one IEEE-rounded f32
 * operation and every f64 operation one IEEE-rounded f64 operation.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ==== threads =================================================================================================== */

/* The oracle runs single-threaded unless a caller (the benchmark's all-cores CPU baseline) asks for more.  Threads
 * only split independent outputs (the rows of a projection, the heads of an attention): every output is computed by
 * the same loop in the same order whatever the thread count, so the results do not depend on it.  Built without
 * OpenMP, the pragmas are ignored and the oracle stays single-threaded. */
static int g_threads = 1;

int ora_set_threads(int n) {
#ifdef _OPENMP
    g_threads = n < 1 ? 1 : n;
#else
    (void)n;
    g_threads = 1;
#endif
    return g_threads;
}

int ora_host_cores(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }

/* ==== Q8_0 matrices ============================================================================================= */

/* qwen_emit docs, struct Q8Ref: a Q8_0 weight is int8 quants plus one f32 scale per 32 inputs,
 * W[o][t] = quants[o*in + t] * scales[o*nb + t/32] with nb = in/32. */
double ora_q8_weight(const int8_t *q, const float *s, int64_t k, int64_t o, int64_t t) {
    int64_t nb = k / ORA_QBLOCK;
    return (double)q[o * k + t] * (double)s[o * nb + t / ORA_QBLOCK];
}

void ora_q8_dequant(const int8_t *q, const float *s, int64_t n, int64_t k, double *w) {
    for (int64_t o = 0; o < n; ++o)
        for (int64_t t = 0; t < k; ++t) w[o * k + t] = ora_q8_weight(q, s, k, o, t);
}

/* qwen_emit docs, emit_moe_forward: the dequant-in-kernel product of an f32 activation by int8 weights with an f64
 * accumulator; forward_shim.rs, ForwardShim::numerics (Q8MatKind::Dequant: no activation quantized).
 * y[o] = sum_t W[o][t] * x[t], every term and the sum in f64. */
void ora_gemv_f32act(const int8_t *q, const float *s, int64_t n, int64_t k, const float *x, double *y) {
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1 && n * k >= (1 << 16))
    for (int64_t o = 0; o < n; ++o) {
        double acc = 0.0;
        for (int64_t t = 0; t < k; ++t) acc += ora_q8_weight(q, s, k, o, t) * (double)x[t];
        y[o] = acc;
    }
}

/* ==== rounding-boundary probe (test support) ====================================================================
 * The one-word rule decides each word by rounding x/d; when a value lies within an f32 rounding error of a half-step
 * boundary, a computation that reaches the same value by another summation order may round it the other way, and
 * both words are results of the rule.  The probe lets a test see those decisions and take the other one: armed for a
 * site, it follows that site's next activation row through every one-word quantization of it, records for each value
 * the signed distance of x/d from the nearest rounding boundary in steps (sign = the direction of that boundary), and
 * adds the requested deltas to chosen words.  Sites: ORA_PROBE_MOE_INPUT, the input row of the next ora_moe_row call
 * (which the router and every expert read); ORA_PROBE_ATTN_OUT, the attention output row that the next
 * ora_decode_layer's O projection reads.  Unarmed (the default) it changes nothing. */
static int g_probe_armed, g_probe_site;
static const float *g_probe_src;
static double *g_probe_margin;
static int g_probe_recorded;
static int64_t g_flip_idx[ORA_MAX_FLIPS];
static int g_flip_delta[ORA_MAX_FLIPS];
static int g_nflip;

void ora_probe_arm(int site, double *margins, const int64_t *flip_idx, const int32_t *flip_delta, int nflip) {
    g_probe_armed = 1;
    g_probe_site = site;
    g_probe_src = NULL;
    g_probe_margin = margins;
    g_probe_recorded = 0;
    g_nflip = nflip < 0 ? 0 : (nflip > ORA_MAX_FLIPS ? ORA_MAX_FLIPS : nflip);
    for (int i = 0; i < g_nflip; ++i) {
        g_flip_idx[i] = flip_idx[i];
        g_flip_delta[i] = flip_delta[i];
    }
}

/* lane/mod.rs module docs ("llama.cpp's one int8 word") and forward_shim.rs, ForwardShim::activation
 * (QuantFormat::OneWord): an activation read by a Q8_0 product is one int8 word per value plus one f32 scale per
 * 32-value block.  The pages do not print the rule; the reading taken (the usual one for that format):
 *   amax = max |x| over the block;  d = amax / 127 (one f32 division);
 *   q = round-half-away-from-zero(x / d) (one f32 division), clamped to [-127, 127];  amax = 0 gives d = 0, q = 0. */
void ora_quantize(const float *x, int64_t n, int8_t *xq, float *xs) {
    for (int64_t b = 0; b < n / ORA_QBLOCK; ++b) {
        const float *v = x + b * ORA_QBLOCK;
        float amax = 0.0f;
        for (int t = 0; t < ORA_QBLOCK; ++t) {
            float a = fabsf(v[t]);
            if (a > amax) amax = a;
        }
        float d = amax / 127.0f;
        xs[b] = d;
        for (int t = 0; t < ORA_QBLOCK; ++t) {
            int8_t w = 0;
            double margin = 0.5;
            if (d != 0.0f) {
                float qv = v[t] / d;
                float r = roundf(qv);
                double off = (double)qv - (double)r;
                margin = off >= 0.0 ? 0.5 - off : -(0.5 + off);
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                w = (int8_t)r;
            }
            xq[b * ORA_QBLOCK + t] = w;
            if (x == g_probe_src && g_probe_margin && !g_probe_recorded) g_probe_margin[b * ORA_QBLOCK + t] = margin;
        }
    }
    if (x == g_probe_src) {
        g_probe_recorded = 1;
        for (int i = 0; i < g_nflip; ++i)
            if (g_flip_idx[i] >= 0 && g_flip_idx[i] < n) {
                int w = xq[g_flip_idx[i]] + g_flip_delta[i];
                xq[g_flip_idx[i]] = (int8_t)(w > 127 ? 127 : (w < -127 ? -127 : w));
            }
    }
}

/* The int32 dot of one weight block with one activation block: exact integer arithmetic. */
void ora_blockdots(const int8_t *q, int64_t n, int64_t k, const int8_t *xq, int32_t *dots) {
    int64_t nb = k / ORA_QBLOCK;
    for (int64_t o = 0; o < n; ++o)
        for (int64_t b = 0; b < nb; ++b) {
            int32_t acc = 0;
            for (int t = 0; t < ORA_QBLOCK; ++t)
                acc += (int32_t)q[o * k + b * ORA_QBLOCK + t] * (int32_t)xq[b * ORA_QBLOCK + t];
            dots[o * nb + b] = acc;
        }
}

/* Int8-activation product (Q8MatKind::Int8Act): y[o] = sum_b s_w[o,b] * s_x[b] * D[o,b], the block dots exact and the
 * scaled sum in f64. */
void ora_gemv_int8act(const int8_t *q, const float *s, int64_t n, int64_t k, const int8_t *xq, const float *xs,
                      double *y) {
    int64_t nb = k / ORA_QBLOCK;
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1 && n * k >= (1 << 16))
    for (int64_t o = 0; o < n; ++o) {
        double acc = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            int32_t dot;
            ora_blockdots(q + o * k + b * ORA_QBLOCK, 1, ORA_QBLOCK, xq + b * ORA_QBLOCK, &dot);
            acc += (double)s[o * nb + b] * (double)xs[b] * (double)dot;
        }
        y[o] = acc;
    }
}

/* The two-word activation (lane/mod.rs module docs: "a two-word ~14-bit int8 activation (the default)";
 * forward_shim.rs, ForwardShim::activation: Q8MatKind::TwoPassInt8 -> QuantFormat::TwoWords; lane/arena.rs,
 * array_bytes and quant_parts: a quantized array is its words, then its low words under two words, then one f32 scale
 * a 32-value block).  The pages give the parts, not the rule.  The reading taken: the high word and the scale are the
 * one-word rule's, and the low word holds what the high word leaves, in 128ths of the scale:
 *   t = x / d (one f32 division, d = amax/127 as above);  hi = round-half-away(t) clamped to +-127;
 *   lo = round-half-away(128 (t - hi))   (t - hi and the product by 128 are exact in f32; |lo| <= 64)
 * so x ~ d (hi + lo/128) = (d/128)(128 hi + lo), a signed integer of 14 magnitude bits (|128 hi + lo| <= 16320)
 * on the block's one scale. */
void ora_quantize2(const float *x, int64_t n, int8_t *hi, int8_t *lo, float *xs) {
    for (int64_t b = 0; b < n / ORA_QBLOCK; ++b) {
        const float *v = x + b * ORA_QBLOCK;
        float amax = 0.0f;
        for (int t = 0; t < ORA_QBLOCK; ++t) {
            float a = fabsf(v[t]);
            if (a > amax) amax = a;
        }
        float d = amax / 127.0f;
        xs[b] = d;
        for (int t = 0; t < ORA_QBLOCK; ++t) {
            int8_t wh = 0, wl = 0;
            if (d != 0.0f) {
                float q = v[t] / d;
                float r = roundf(q);
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                float f = roundf((q - r) * 128.0f);
                if (f > 127.0f) f = 127.0f;
                if (f < -127.0f) f = -127.0f;
                wh = (int8_t)r;
                wl = (int8_t)f;
            }
            hi[b * ORA_QBLOCK + t] = wh;
            lo[b * ORA_QBLOCK + t] = wl;
        }
    }
}

/* The two-word product: per block the exact integer 128 D[o,b](hi) + D[o,b](lo) of the two words' int32 dots, so
 * y[o] = sum_b s_w[o,b] * s_x[b] / 128 * (128 D_hi + D_lo), in f64. */
void ora_gemv_int8act2(const int8_t *q, const float *s, int64_t n, int64_t k, const int8_t *hi, const int8_t *lo,
                       const float *xs, double *y) {
    int64_t nb = k / ORA_QBLOCK;
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1 && n * k >= (1 << 16))
    for (int64_t o = 0; o < n; ++o) {
        double acc = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            int32_t dh, dl;
            ora_blockdots(q + o * k + b * ORA_QBLOCK, 1, ORA_QBLOCK, hi + b * ORA_QBLOCK, &dh);
            ora_blockdots(q + o * k + b * ORA_QBLOCK, 1, ORA_QBLOCK, lo + b * ORA_QBLOCK, &dl);
            acc += (double)s[o * nb + b] * (double)xs[b] / 128.0 * (128.0 * (double)dh + (double)dl);
        }
        y[o] = acc;
    }
}

void ora_gemv(int mode, const int8_t *q, const float *s, int64_t n, int64_t k, const float *x, double *y) {
    if (mode == 0) {
        ora_gemv_f32act(q, s, n, k, x, y);
        return;
    }
    if (mode == 2) {
        int8_t *hi = (int8_t *)malloc((size_t)(k > 0 ? k : 1));
        int8_t *lo = (int8_t *)malloc((size_t)(k > 0 ? k : 1));
        float *xs = (float *)malloc(sizeof(float) * (size_t)(k / ORA_QBLOCK + 1));
        ora_quantize2(x, k, hi, lo, xs);
        ora_gemv_int8act2(q, s, n, k, hi, lo, xs, y);
        free(hi);
        free(lo);
        free(xs);
        return;
    }
    int8_t *xq = (int8_t *)malloc((size_t)(k > 0 ? k : 1));
    float *xs = (float *)malloc(sizeof(float) * (size_t)(k / ORA_QBLOCK + 1));
    ora_quantize(x, k, xq, xs);
    ora_gemv_int8act(q, s, n, k, xq, xs, y);
    free(xq);
    free(xs);
}

/* ==== residual add + RMSNorm ==================================================================================== */

/* forward_shim.rs module docs and ForwardShim::fits (AddNorm): the sum is written out whole and the RMS norm of the
 * whole sum follows; ForwardShim::supports (CompensatedResidual refused): the residual is summed in f32,
 * uncompensated; kernel_refusal: an RMS norm scales by its weight and never shifts.  Reading: eps inside the root,
 * added to the mean of squares.
 *   s = fl32(a + b)          y = s / sqrt(mean(s^2) + eps) * w      (the norm in f64) */
void ora_add_rmsnorm(const float *a, const float *b, const float *w, int64_t rows, int64_t d, float eps, float *sum,
                     double *y) {
    float *row = (float *)malloc(sizeof(float) * (size_t)(d > 0 ? d : 1));
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t i = 0; i < d; ++i) {
            float v = a[r * d + i];
            if (b) v = v + b[r * d + i];
            row[i] = v;
            if (sum) sum[r * d + i] = v;
        }
        double ms = 0.0;
        for (int64_t i = 0; i < d; ++i) ms += (double)row[i] * (double)row[i];
        ms /= (double)d;
        double inv = 1.0 / sqrt(ms + (double)eps);
        for (int64_t i = 0; i < d; ++i) y[r * d + i] = (double)row[i] * inv * (double)w[i];
    }
    free(row);
}

/* ==== router, gating, mixture =================================================================================== */

void ora_softmax(const double *l, int64_t n, double *p) {
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i)
        if (l[i] > m) m = l[i];
    double z = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        p[i] = exp(l[i] - m);
        z += p[i];
    }
    for (int64_t i = 0; i < n; ++i) p[i] /= z;
}

/* The k largest values in descending order, equal values taken lower index first. */
void ora_topk(const double *p, int64_t n, int k, int32_t *ids) {
    unsigned char *taken = (unsigned char *)calloc((size_t)(n > 0 ? n : 1), 1);
    for (int j = 0; j < k; ++j) {
        int64_t best = -1;
        for (int64_t i = 0; i < n; ++i)
            if (!taken[i] && (best < 0 || p[i] > p[best])) best = i;
        taken[best] = 1;
        ids[j] = (int32_t)best;
    }
    free(taken);
}

/* forward_shim.rs, kernel_refusal (Moe arms: refused unless the router is a softmax weighting its experts' outputs and
 * renormalizes the kept experts' weights); qwen_emit docs, emit_moe_forward (softmax, keep K, renormalize).
 * Reading: the kept experts are the K largest probabilities, i.e. the K largest logits (selected on the logits, the
 * softmax being strictly increasing), in descending order with ties to the lower index; g_j = p_j / sum_kept p. */
void ora_route(const double *logits, int64_t experts, int k, int32_t *ids, double *gates) {
    double *p = (double *)malloc(sizeof(double) * (size_t)experts);
    ora_softmax(logits, experts, p);
    ora_topk(logits, experts, k, ids);
    double z = 0.0;
    for (int j = 0; j < k; ++j) z += p[ids[j]];
    for (int j = 0; j < k; ++j) gates[j] = p[ids[j]] / z;
    free(p);
}

/* forward_shim.rs, kernel_refusal (only SwiGLU experts): silu(z) = z / (1 + e^-z); the expert's hidden value is
 * silu(gate . x) * (up . x). */
double ora_silu(double z) { return z / (1.0 + exp(-z)); }

/* lane_link.rs, Link::prim (Moe: Router::F32, a router whose operand is values rather than quantized checkpoint rows):
 * the router's logits as a product of f32 values by the f32 activation.  Every term and the sum in f64. */
void ora_gemv_f32w(const float *w, int64_t n, int64_t k, const float *x, double *y) {
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1 && n * k >= (1 << 16))
    for (int64_t o = 0; o < n; ++o) {
        double acc = 0.0;
        for (int64_t t = 0; t < k; ++t) acc += (double)w[o * k + t] * (double)x[t];
        y[o] = acc;
    }
}

/* qwen_emit docs, MoeWeights (router [E,d]; gate/up [E*dff,d] with expert e at row e*dff; down [E*d,dff] with expert e
 * at row e*d) and emit_moe_forward (router product, softmax top-K renormalized, each expert's SwiGLU at an
 * expert-indexed base, weighted combine).  In the int8 modes every Q8_0 projection reads its activation quantized
 * (forward_shim.rs, ForwardShim::activation: operand 0 of a Q8_0 product or a mixture); the hidden row is held in f32
 * before the down product reads it.
 * An f32 router (lane_link.rs, Link::prim: Router::F32) is a product of values, not of quantized rows: it reads the
 * f32 activation in every mode.
 * A shared expert (lane_link.rs, Link::class_launch: SharedExpertFusion, the mixture with the shared expert's gated pair
 * and down product in one launch; SharedExperts {wg, wu, wd, dff}) is a SwiGLU feed-forward every row passes through,
 * unweighted: its output is added to the weighted sum of the kept experts, after them. */
void ora_moe_row(int mode, const ora_moe *m, const float *x, const float *residual, double *logits, int32_t *ids,
                 double *gates, double *hidden, double *expert_out, double *y, double *shared_hidden,
                 double *shared_out) {
    const int64_t d = m->d, dff = m->dff, E = m->experts;
    const int K = m->k;
    if (g_probe_armed && g_probe_site == ORA_PROBE_MOE_INPUT) {  /* this row's input takes the probe (test support) */
        g_probe_armed = 0;
        g_probe_src = x;
    }
    double *l = (double *)malloc(sizeof(double) * (size_t)E);
    if (m->router_f32)
        ora_gemv_f32w(m->router_f32, E, d, x, l);
    else
        ora_gemv(mode, m->router.q, m->router.s, E, d, x, l);
    if (logits) memcpy(logits, l, sizeof(double) * (size_t)E);
    double g[64];
    int32_t id[64];
    ora_route(l, E, K, id, g);
    double *gv = (double *)malloc(sizeof(double) * (size_t)dff);
    double *uv = (double *)malloc(sizeof(double) * (size_t)dff);
    float *h32 = (float *)malloc(sizeof(float) * (size_t)dff);
    double *yj = (double *)malloc(sizeof(double) * (size_t)d);
    double *acc = (double *)calloc((size_t)d, sizeof(double));
    const int64_t nbd = d / ORA_QBLOCK, nbf = dff / ORA_QBLOCK;
    for (int j = 0; j < K; ++j) {
        const int64_t e = id[j];
        ora_gemv(mode, m->gate.q + e * dff * d, m->gate.s + e * dff * nbd, dff, d, x, gv);
        ora_gemv(mode, m->up.q + e * dff * d, m->up.s + e * dff * nbd, dff, d, x, uv);
        for (int64_t i = 0; i < dff; ++i) {
            double h = ora_silu(gv[i]) * uv[i];
            if (hidden) hidden[j * dff + i] = h;
            h32[i] = (float)h;
        }
        ora_gemv(mode, m->down.q + e * d * dff, m->down.s + e * d * nbf, d, dff, h32, yj);
        for (int64_t o = 0; o < d; ++o) {
            if (expert_out) expert_out[j * d + o] = yj[o];
            acc[o] += g[j] * yj[o];
        }
    }
    if (m->sdff > 0) {  /* the shared expert, after the kept experts */
        const int64_t sdff = m->sdff;
        double *sg = (double *)malloc(sizeof(double) * (size_t)sdff);
        double *su = (double *)malloc(sizeof(double) * (size_t)sdff);
        float *sh32 = (float *)malloc(sizeof(float) * (size_t)sdff);
        ora_gemv(mode, m->sgate.q, m->sgate.s, sdff, d, x, sg);
        ora_gemv(mode, m->sup.q, m->sup.s, sdff, d, x, su);
        for (int64_t i = 0; i < sdff; ++i) {
            double h = ora_silu(sg[i]) * su[i];
            if (shared_hidden) shared_hidden[i] = h;
            sh32[i] = (float)h;
        }
        ora_gemv(mode, m->sdown.q, m->sdown.s, d, sdff, sh32, yj);
        for (int64_t o = 0; o < d; ++o) {
            if (shared_out) shared_out[o] = yj[o];
            acc[o] += yj[o];
        }
        free(sg);
        free(su);
        free(sh32);
    }
    for (int64_t o = 0; o < d; ++o) y[o] = (residual ? (double)residual[o] : 0.0) + acc[o];
    for (int j = 0; j < K; ++j) {
        ids[j] = id[j];
        gates[j] = g[j];
    }
    free(l);
    free(gv);
    free(uv);
    free(h32);
    free(yj);
    free(acc);
    if (g_probe_src == x) g_probe_src = NULL;
}

/* lane_link.rs, Link::class_launch (MoeTokenSort) and lane/arena.rs, scratch (a chunk's choices counted per expert,
 * their offsets and per-expert lists): a counting sort of the chunk's choices by expert, stable in choice order. */
void ora_group(const int32_t *ids, int64_t rows, int k, int64_t experts, int32_t *counts, int32_t *offsets,
               int32_t *lists) {
    const int64_t n = rows * k;
    for (int64_t e = 0; e < experts; ++e) counts[e] = 0;
    for (int64_t c = 0; c < n; ++c) counts[ids[c]] += 1;
    offsets[0] = 0;
    for (int64_t e = 0; e < experts; ++e) offsets[e + 1] = offsets[e] + counts[e];
    for (int64_t e = 0; e < experts; ++e) {
        int32_t at = offsets[e];
        for (int64_t c = 0; c < n; ++c)
            if (ids[c] == e) lists[at++] = (int32_t)c;
    }
}

/* ==== decode step ================================================================================================ */

/* Per-head RMS norm (the QK-norm of qwen_emit docs, emit_qwen30b_generate): y = x / sqrt(mean(x^2) + eps) * w. */
void ora_rmsnorm_head(const double *x, const float *w, int64_t n, float eps, double *y) {
    double ms = 0.0;
    for (int64_t i = 0; i < n; ++i) ms += x[i] * x[i];
    double inv = 1.0 / sqrt(ms / (double)n + (double)eps);
    for (int64_t i = 0; i < n; ++i) y[i] = x[i] * inv * (double)w[i];
}

/* forward_shim.rs, kernel_refusal (Rope arms: a full rotary, every dimension turned, hd = 2*half).  Reading: the pairs
 * are the two halves (i, i + hd/2), angle = pos * theta^(-2i/hd). */
void ora_rope(double *x, int64_t hd, int64_t pos, double theta) {
    const int64_t half = hd / 2;
    for (int64_t i = 0; i < half; ++i) {
        double ang = (double)pos * pow(theta, -2.0 * (double)i / (double)hd);
        double c = cos(ang), s = sin(ang);
        double a = x[i], b = x[i + half];
        x[i] = a * c - b * s;
        x[i + half] = a * s + b * c;
    }
}

/* forward_shim.rs, kernel_refusal (Attention arms: scores scaled by 1/sqrt(hd), no mask, window, sink or cap); one
 * query over `len` cached rows: out = sum_p softmax_p(q . k_p / sqrt(hd)) v_p. */
void ora_attention(const double *q, const float *kc, const float *vc, int64_t len, int64_t hd, double *out) {
    double *sc = (double *)malloc(sizeof(double) * (size_t)len);
    double *p = (double *)malloc(sizeof(double) * (size_t)len);
    const double scale = 1.0 / sqrt((double)hd);
    for (int64_t t = 0; t < len; ++t) {
        double acc = 0.0;
        for (int64_t i = 0; i < hd; ++i) acc += q[i] * (double)kc[t * hd + i];
        sc[t] = acc * scale;
    }
    ora_softmax(sc, len, p);
    for (int64_t i = 0; i < hd; ++i) {
        double acc = 0.0;
        for (int64_t t = 0; t < len; ++t) acc += p[t] * (double)vc[t * hd + i];
        out[i] = acc;
    }
    free(sc);
    free(p);
}

/* The greedy next token: the first index of the largest logit. */
int64_t ora_argmax(const double *x, int64_t n) {
    int64_t best = 0;
    for (int64_t i = 1; i < n; ++i)
        if (x[i] > x[best]) best = i;
    return best;
}

static void to_f32(const double *x, int64_t n, float *y) {
    for (int64_t i = 0; i < n; ++i) y[i] = (float)x[i];
}

/* qwen_emit docs, emit_qwen30b_generate: RMSNorm -> Q/K/V -> per-head QK-norm + RoPE -> attention over the KV cache ->
 * O-proj -> residual -> RMSNorm -> mixture -> residual, per layer; then the LM head and the greedy token.  The
 * residual stream and the caches are f32 (forward_shim.rs, ForwardShim::supports: CompensatedResidual and
 * KvCacheQuant refused); every projection reads an f32 activation (quantized in mode 1).
 *
 * One layer: h is the residual stream entering layer l (for the first layer the token's embedding row, which is normed
 * with no residual added); on return it holds the stream leaving the layer, h + o and then + the mixture, each sum one
 * f32 add.  The layer's key and value rows are written into the caches at `pos`.  router_logits (NULL or [experts])
 * receives the router's logits. */
void ora_decode_layer(int mode, const ora_model *m, int64_t l, int64_t pos, float *h, double *router_logits) {
    const int64_t d = m->d, H = m->heads, KV = m->kv_heads, hd = m->hd, ctx = m->ctx;
    const int64_t group = H / KV;
    double *n64 = (double *)malloc(sizeof(double) * (size_t)d);
    float *x32 = (float *)malloc(sizeof(float) * (size_t)(H * hd > d ? H * hd : d));
    double *q = (double *)malloc(sizeof(double) * (size_t)(H * hd));
    double *k = (double *)malloc(sizeof(double) * (size_t)(KV * hd));
    double *v = (double *)malloc(sizeof(double) * (size_t)(KV * hd));
    double *att = (double *)malloc(sizeof(double) * (size_t)(H * hd));
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    float *o32 = (float *)malloc(sizeof(float) * (size_t)d);
    float *moe_out = (float *)malloc(sizeof(float) * (size_t)d);
    int32_t ids[64];
    double gates[64];

    /* attention half */
    ora_add_rmsnorm(h, NULL, m->attn_norm[l], 1, d, m->eps, NULL, n64);
    to_f32(n64, d, x32);
    ora_gemv(mode, m->wq[l].q, m->wq[l].s, H * hd, d, x32, q);
    ora_gemv(mode, m->wk[l].q, m->wk[l].s, KV * hd, d, x32, k);
    ora_gemv(mode, m->wv[l].q, m->wv[l].s, KV * hd, d, x32, v);
    for (int64_t hh = 0; hh < H; ++hh) {
        ora_rmsnorm_head(q + hh * hd, m->q_norm[l], hd, m->eps, q + hh * hd);
        ora_rope(q + hh * hd, hd, pos, m->rope_theta);
    }
    for (int64_t g = 0; g < KV; ++g) {
        ora_rmsnorm_head(k + g * hd, m->k_norm[l], hd, m->eps, k + g * hd);
        ora_rope(k + g * hd, hd, pos, m->rope_theta);
        float *kr = m->k_cache[l] + (g * ctx + pos) * hd;
        float *vr = m->v_cache[l] + (g * ctx + pos) * hd;
        for (int64_t i = 0; i < hd; ++i) {
            kr[i] = (float)k[g * hd + i];
            vr[i] = (float)v[g * hd + i];
        }
    }
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1)
    for (int64_t hh = 0; hh < H; ++hh) {
        const int64_t g = hh / group;
        ora_attention(q + hh * hd, m->k_cache[l] + g * ctx * hd, m->v_cache[l] + g * ctx * hd, pos + 1, hd,
                      att + hh * hd);
    }
    to_f32(att, H * hd, x32);
    if (g_probe_armed && g_probe_site == ORA_PROBE_ATTN_OUT) {  /* the O projection's input takes the probe */
        g_probe_armed = 0;
        g_probe_src = x32;
    }
    ora_gemv(mode, m->wo[l].q, m->wo[l].s, d, H * hd, x32, o);
    if (g_probe_src == x32) g_probe_src = NULL;
    to_f32(o, d, o32);
    /* feed-forward half: the norm of h + o (the sum kept as the residual) feeds the mixture */
    ora_add_rmsnorm(h, o32, m->ffn_norm[l], 1, d, m->eps, h, n64);
    to_f32(n64, d, x32);
    ora_moe mo = m->moe;
    mo.router = m->router[l];
    mo.gate = m->gate[l];
    mo.up = m->up[l];
    mo.down = m->down[l];
    mo.router_f32 = m->router_f32 ? m->router_f32[l] : NULL;
    if (m->sgate && mo.sdff > 0) {
        mo.sgate = m->sgate[l];
        mo.sup = m->sup[l];
        mo.sdown = m->sdown[l];
    } else {
        mo.sdff = 0;
    }
    ora_moe_row(mode, &mo, x32, NULL, router_logits, ids, gates, NULL, NULL, y, NULL, NULL);
    to_f32(y, d, moe_out);
    for (int64_t i = 0; i < d; ++i) h[i] = h[i] + moe_out[i];
    free(n64);
    free(x32);
    free(q);
    free(k);
    free(v);
    free(att);
    free(o);
    free(y);
    free(o32);
    free(moe_out);
}

/* The first `layers` layers from the token's embedding row. */
static void run_layers(int mode, const ora_model *m, int64_t tok, int64_t pos, int64_t layers, float *h) {
    memcpy(h, m->embed + tok * m->d, sizeof(float) * (size_t)m->d);
    for (int64_t l = 0; l < layers; ++l) ora_decode_layer(mode, m, l, pos, h, NULL);
}

/* The step's end (qwen_emit docs, emit_qwen30b_generate): the final RMSNorm of the residual stream h, the LM head and
 * the greedy token. */
int64_t ora_decode_final(int mode, const ora_model *m, const float *h, double *logits) {
    const int64_t d = m->d;
    double *n64 = (double *)malloc(sizeof(double) * (size_t)d);
    float *x32 = (float *)malloc(sizeof(float) * (size_t)d);
    ora_add_rmsnorm(h, NULL, m->final_norm, 1, d, m->eps, NULL, n64);
    to_f32(n64, d, x32);
    ora_gemv(mode, m->lm_head.q, m->lm_head.s, m->vocab, d, x32, logits);
    free(n64);
    free(x32);
    return ora_argmax(logits, m->vocab);
}

int64_t ora_decode_step(int mode, const ora_model *m, int64_t tok, int64_t pos, double *logits) {
    float *h = (float *)malloc(sizeof(float) * (size_t)m->d);
    run_layers(mode, m, tok, pos, m->layers, h);
    const int64_t next = ora_decode_final(mode, m, h, logits);
    free(h);
    return next;
}

void ora_decode_layers(int mode, const ora_model *m, int64_t tok, int64_t pos, int64_t layers, double *hidden_out) {
    const int64_t d = m->d;
    float *h = (float *)malloc(sizeof(float) * (size_t)d);
    run_layers(mode, m, tok, pos, layers, h);
    for (int64_t i = 0; i < d; ++i) hidden_out[i] = (double)h[i];
    free(h);
}
