/*
 * CPU oracle of the Q8_0 mixture-of-experts decode step — TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may load or call this library.  It shares
 * no code with the CUDA path: it is a plain, slow restatement in C of what the pages define (single-threaded unless
 * ora_set_threads asks for more), in f64
 * wherever the pages do not fix another precision.  Each function names the passage it follows.
 *
 * Pages cited (their titles):
 *   qwen_emit  — "logicaffeine_compile/codegen_cuda/qwen_emit" module docs (Q8Ref, MoeWeights, Q8MatKind,
 *                emit_moe_forward, emit_qwen30b_generate, moe_dp4a_kernels)
 *   forward_shim.rs — "codegen_cuda/forward_shim.rs" (module docs, kernel_refusal, ForwardShim::supports/numerics)
 *   lane_link.rs    — "codegen_cuda/lane_link.rs" (Link::prim, Link::class_launch)
 *   lane/mod.rs     — "codegen_cuda/lane/mod.rs" (module docs: the knobs and numerics)
 *   lane/arena.rs   — "codegen_cuda/lane/arena.rs" (scratch: the mixture's choices, weights and hidden rows)
 *
 * Parity pins: every function here is pinned by tests marked "not gpu" against hand-worked values, closed forms,
 * invariants and exact brute force; none is "parity unpinned".
 */
#ifndef ORACLE_H
#define ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORA_QBLOCK 32

/* Threads the oracle may use (1 unless set; the results do not depend on it) and the host's online cores. */
int ora_set_threads(int n);
int ora_host_cores(void);

/* ---- Q8_0 matrices and projections ---------------------------------------------------------------------------- */
double ora_q8_weight(const int8_t *q, const float *s, int64_t k, int64_t o, int64_t t);
void ora_q8_dequant(const int8_t *q, const float *s, int64_t n, int64_t k, double *w);
void ora_gemv_f32act(const int8_t *q, const float *s, int64_t n, int64_t k, const float *x, double *y);
void ora_quantize(const float *x, int64_t n, int8_t *xq, float *xs);
void ora_blockdots(const int8_t *q, int64_t n, int64_t k, const int8_t *xq, int32_t *dots);
void ora_gemv_int8act(const int8_t *q, const float *s, int64_t n, int64_t k, const int8_t *xq, const float *xs,
                      double *y);
/* The two-word activation: high words, low words (128ths of the scale) and one scale per 32-value block. */
void ora_quantize2(const float *x, int64_t n, int8_t *hi, int8_t *lo, float *xs);
void ora_gemv_int8act2(const int8_t *q, const float *s, int64_t n, int64_t k, const int8_t *hi, const int8_t *lo,
                       const float *xs, double *y);
/* mode 0: f32 activations, f64 sums; mode 1: x quantized to one int8 word per value, then mode-1 sums; mode 2: x
 * quantized to two words per value, then the two-word sums. */
void ora_gemv(int mode, const int8_t *q, const float *s, int64_t n, int64_t k, const float *x, double *y);

/* ---- residual add + RMSNorm ----------------------------------------------------------------------------------- */
void ora_add_rmsnorm(const float *a, const float *b, const float *w, int64_t rows, int64_t d, float eps, float *sum,
                     double *y);

/* ---- router, gating, mixture ---------------------------------------------------------------------------------- */
void ora_softmax(const double *l, int64_t n, double *p);
void ora_topk(const double *p, int64_t n, int k, int32_t *ids);
void ora_route(const double *logits, int64_t experts, int k, int32_t *ids, double *gates);
double ora_silu(double z);

typedef struct {
    const int8_t *q;
    const float *s;
} ora_q8;

typedef struct {
    int64_t d, dff, experts;
    int k;
    ora_q8 router; /* [experts, d] */
    ora_q8 gate;   /* [experts*dff, d], expert e at row e*dff */
    ora_q8 up;     /* [experts*dff, d] */
    ora_q8 down;   /* [experts*d, dff], expert e at row e*d */
    const float *router_f32; /* NULL, or a router of f32 values [experts, d] used in place of `router` */
    int64_t sdff;            /* 0, or the shared expert's hidden width */
    ora_q8 sgate, sup;       /* the shared expert: [sdff, d] each */
    ora_q8 sdown;            /* [d, sdff] */
} ora_moe;

/* y[o] = sum_t w[o][t] * x[t] for a matrix of f32 values, every term and the sum in f64. */
void ora_gemv_f32w(const float *w, int64_t n, int64_t k, const float *x, double *y);
/* One row through the mixture; every output pointer but ids/gates/y may be NULL.  With a shared expert, shared_hidden
 * [sdff] and shared_out [d] receive its hidden row and its output. */
void ora_moe_row(int mode, const ora_moe *m, const float *x, const float *residual, double *logits, int32_t *ids,
                 double *gates, double *hidden, double *expert_out, double *y, double *shared_hidden,
                 double *shared_out);
/* Test support: the next activation row of `site` is probed through every one-word quantization of it — margins (may
 * be NULL) receives, per value, the signed distance of x/d from the nearest rounding boundary in steps (sign = that
 * boundary's direction, a signed zero for an exact tie; 0.5 for a value of an all-zero block), and each word flip_idx[i] gets flip_delta[i] added
 * (clamped to +-127).  Sites: the next ora_moe_row call's input row, or the attention output row that the next
 * ora_decode_layer's O projection reads.  One-shot; unarmed, nothing changes. */
#define ORA_MAX_FLIPS 8
#define ORA_PROBE_MOE_INPUT 0
#define ORA_PROBE_ATTN_OUT 1
void ora_probe_arm(int site, double *margins, const int64_t *flip_idx, const int32_t *flip_delta, int nflip);
/* Choices of a chunk grouped by expert: counts[e], offsets[e] (offsets[experts] = rows*k) and the choice indices
 * r*k+j of each expert in ascending order. */
void ora_group(const int32_t *ids, int64_t rows, int k, int64_t experts, int32_t *counts, int32_t *offsets,
               int32_t *lists);

/* ---- the decode step ------------------------------------------------------------------------------------------ */
void ora_rmsnorm_head(const double *x, const float *w, int64_t n, float eps, double *y);
void ora_rope(double *x, int64_t hd, int64_t pos, double theta);
void ora_attention(const double *q, const float *kc, const float *vc, int64_t len, int64_t hd, double *out);
int64_t ora_argmax(const double *x, int64_t n);

typedef struct {
    int64_t layers, d, heads, kv_heads, hd, vocab, ctx;
    float eps;
    double rope_theta;
    ora_moe moe;                           /* shapes only; per-layer weights below */
    const float *embed;                    /* [vocab, d] */
    const float *const *attn_norm;         /* [layers] -> [d] */
    const float *const *ffn_norm;          /* [layers] -> [d] */
    const float *const *q_norm;            /* [layers] -> [hd] */
    const float *const *k_norm;            /* [layers] -> [hd] */
    const float *final_norm;               /* [d] */
    const ora_q8 *wq, *wk, *wv, *wo;       /* [layers] */
    const ora_q8 *router, *gate, *up, *down; /* [layers] */
    const float *const *router_f32;        /* NULL, or [layers] -> f32 router values [experts, d] */
    const ora_q8 *sgate, *sup, *sdown;     /* NULL, or [layers]: the shared expert (moe.sdff wide) */
    ora_q8 lm_head;                        /* [vocab, d] */
    float *const *k_cache;                 /* [layers] -> [kv_heads, ctx, hd] */
    float *const *v_cache;                 /* [layers] -> [kv_heads, ctx, hd] */
} ora_model;

/* One token at `pos`: writes the new key/value rows into the caches, fills logits[vocab] and returns the argmax. */
int64_t ora_decode_step(int mode, const ora_model *m, int64_t tok, int64_t pos, double *logits);
/* Layer l alone: h [d] is the residual stream entering the layer (the embedding row for the first layer) and holds the
 * stream leaving it on return; the layer's key/value rows are written at `pos`; router_logits may be NULL. */
void ora_decode_layer(int mode, const ora_model *m, int64_t l, int64_t pos, float *h, double *router_logits);
/* The step's end from the residual stream h [d] leaving the last layer: final norm, LM head, greedy token. */
int64_t ora_decode_final(int mode, const ora_model *m, const float *h, double *logits);
/* The first `layers` layers of the step only (for a bounded CPU timing sample); returns nothing. */
void ora_decode_layers(int mode, const ora_model *m, int64_t tok, int64_t pos, int64_t layers, double *hidden_out);

#ifdef __cplusplus
}
#endif
#endif
