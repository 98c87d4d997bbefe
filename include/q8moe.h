/*
 * q8moe — C ABI of a GB300 (sm_103a) Q8_0 mixture-of-experts decode step.
 *
 * The calls compute the batch-1 (and small-chunk) decode step of a Q8_0-quantized transformer whose feed-forward block
 * is a sparse mixture of experts.  They follow the pages of the "logicaffeine_compile/codegen_cuda" documentation:
 *   - forward_shim.rs (module docs; kernel_refusal; ForwardShim::supports / numerics / activation),
 *   - lane_link.rs (Link::prim: the Gemv, Norm, Moe, Rope, Attention, ArgMax launch records),
 *   - lane/mod.rs (module docs: the three projection numerics),
 *   - lane/arena.rs (scratch: arrival counters that are zero before and after a launch),
 *   - qwen_emit module docs (Q8Ref, MoeWeights, Q8MatKind, emit_moe_forward, emit_qwen30b_generate).
 *
 * Conventions shared by every call:
 *   - Pointers named as device pointers must be device memory of the current device (or managed memory); host
 *     pointers are named as such.  Every buffer is owned by the caller; the library owns only the workspace and the
 *     decode model's internal buffers and graphs.
 *   - Layouts are dense and row-major.  A Q8_0 matrix of `rows` x `cols` is two arrays: int8 quants q[rows*cols]
 *     (row o at q + o*cols) and f32 block scales s[rows*(cols/32)] (qwen_emit, Q8Ref:
 *     W[o][t] = q[o*cols + t] * s[o*(cols/32) + t/32]).  cols must be a multiple of 32; q must be 32-byte aligned and s
 *     4-byte aligned.
 *   - A quantized activation (one int8 word per value plus one f32 scale per 32-value block; lane/mod.rs module docs,
 *     "llama.cpp's one int8 word") of R rows x C values is q[R*C] int8 and s[R*(C/32)] f32, q 32-byte aligned.
 *     Quantisation rule: d = max|x|/127 over the block; word = round-half-away-from-zero(x/d) clamped to +-127, both
 *     divisions IEEE f32; a block of zeros has d = 0 and zero words.
 *   - The two-word form (lane/mod.rs module docs: "a two-word ~14-bit int8 activation"; lane/arena.rs, array_bytes and
 *     quant_parts: the words, then the low words, then one scale a block) adds low words lo[R*C] int8 (32-byte
 *     aligned): with t = x/d (IEEE f32) and q the word above, lo = round-half-away-from-zero(128 (t - q)), so
 *     x ~ d (q + lo/128); together 128 q + lo is a signed integer of 14 magnitude bits on the block's one scale.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy default stream), allocates nothing,
 *     never synchronizes and never reads device memory back to the host, so every call but the first decode_step can
 *     be captured into a CUDA graph.
 *   - Arguments are checked before any launch.  A bad argument returns Q8_EINVAL (Q8_EUNSUPPORTED for a shape the
 *     kernels refuse, as kernel_refusal does in forward_shim.rs) and launches nothing; q8_last_error() names the
 *     argument.  A CUDA launch error returns Q8_ECUDA.  Errors raised later on the device surface at the caller's next
 *     synchronization as CUDA errors.  A bounded device-side wait that gives up (Q8_ETIMEOUT) is reported only for the
 *     decode model, by q8_model_check; a standalone call whose wait gave up leaves its outputs incomplete and reports
 *     nothing.
 *   - Calls that take a workspace use its scratch and its arrival counters.  Calls sharing one workspace must be
 *     ordered (one stream, or events); two calls that overlap on the device through one workspace race.
 */
#ifndef Q8MOE_H
#define Q8MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define Q8_API __attribute__((visibility("default")))
#else
#define Q8_API
#endif

typedef struct CUstream_st *q8_stream; /* cudaStream_t */

typedef enum {
    Q8_OK = 0,
    Q8_EINVAL = -1,       /* a null, misaligned or out-of-range argument */
    Q8_EUNSUPPORTED = -2, /* a shape the kernels refuse (cols % 32, K outside [1,32], more than 8192 experts, ...) */
    Q8_ECUDA = -3,        /* a CUDA runtime error (launch, capture, allocation at create time) */
    Q8_ETIMEOUT = -4,     /* a bounded device-side wait gave up (reported by q8_model_check) */
    Q8_ENOSPACE = -5      /* the workspace is too small for the call */
} q8_status;

/* The projection numerics (lane/mod.rs module docs; forward_shim.rs, ForwardShim::numerics):
 *   Q8_F32ACT_F64SUM — f32 activations times dequantized int8 weights, each 32-block's f32 partial sum added into an
 *                      f64 accumulator (qwen_emit, emit_moe_forward: "f32 activation x int8 weight, f64 accumulate");
 *   Q8_INT8ACT       — the activation quantized to one int8 word per value; each 32-block's exact int32 dot is
 *                      scaled by both block scales and summed in f32;
 *   Q8_INT8ACT2      — the activation in the two-word form (Q8MatKind::TwoPassInt8 -> QuantFormat::TwoWords, the
 *                      lane's default); each 32-block's exact integer 128 D(words) + D(low words) is scaled by both
 *                      block scales and 1/128 and summed in f32. */
typedef enum { Q8_F32ACT_F64SUM = 0, Q8_INT8ACT = 1, Q8_INT8ACT2 = 2 } q8_mode;

/* A device Q8_0 matrix (see the layout above). */
typedef struct {
    const int8_t *q;
    const float *s;
    int64_t rows, cols;
} q8_mat;

/* A device quantized activation (see the layout above): words q, scales s, and the two-word form's low words lo
 * (read and written only in Q8_INT8ACT2; NULL otherwise). */
typedef struct {
    int8_t *q;
    float *s;
    int8_t *lo;
} q8_act;

/* ---- workspace ------------------------------------------------------------------------------------------------ */
typedef struct q8_ws q8_ws;

/* Allocates a workspace on the current device: `bytes` of scratch (0 picks 64 MiB) plus a zeroed array of arrival
 * counters.  Counters are zero between calls: the last block of a launch to arrive resets them (lane/arena.rs,
 * Scratch: "a counter ... is zero before the launch and left zero by it").  Returns Q8_ECUDA if allocation fails. */
Q8_API int q8_workspace_create(size_t bytes, q8_ws **ws);
Q8_API void q8_workspace_destroy(q8_ws *ws);
Q8_API size_t q8_workspace_bytes(const q8_ws *ws);

/* ---- a1 / K4: quantisation and the residual add + RMSNorm -------------------------------------------------------- */

/* Quantizes x (device f32, rows x cols, cols % 32 == 0) to out (lane_link.rs, Link::prim: the standalone Quant
 * launch); when out->lo is not NULL, to the two-word form. */
Q8_API int q8_quantize(const float *x, int64_t rows, int64_t cols, const q8_act *out, q8_stream stream);

/* Fused residual add + RMSNorm with an int8 epilogue (forward_shim.rs module docs: "a sum and the RMS norm of it ... as
 * one row kernel writing the sum on"; "the activation a Q8_0 projection reads quantized in its producer's epilogue").
 * For each of `rows` rows of d values (device f32):
 *     s = a + b (one f32 add; b may be NULL: s = a)           -> sum_out (may be NULL; may alias a)
 *     y = s / sqrt(mean(s^2) + eps) * w   (the norm in f64, y rounded once to f32)  -> y_out (may be NULL)
 *     yq = quantize(y)                                         -> yq (may be NULL; needs d % 32 == 0; the two-word
 *                                                                 form when yq->lo is not NULL)
 * w is device f32 [d].  At least one output must be given.  eps >= 0. */
Q8_API int add_rmsnorm_q8(const float *a, const float *b, const float *w, int64_t rows, int64_t d, float eps, float *sum_out,
                   float *y_out, const q8_act *yq, q8_stream stream);

/* ---- a2-a4: the Q8_0 projection ----------------------------------------------------------------------------------- */

/* y[r][o] = sum_t W[o][t] * x[r][t] for r < rows (lane_link.rs, Link::prim: Gemv{x, w, y, k, n, m}; qwen_emit, Q8Ref).
 * mode Q8_F32ACT_F64SUM reads x (device f32 [rows][W.cols]); mode Q8_INT8ACT reads xq ([rows][W.cols] words plus
 * scales) and mode Q8_INT8ACT2 xq with its low words, or, when xq is NULL, either quantizes x first into workspace
 * scratch.  y is device f32 [rows][W.rows].  Matrices
 * whose rows under-fill the GPU are cut along k; the partial sums meet in workspace scratch and the last slice to
 * arrive adds them in slice order (lane_link.rs, Link::prim: gemm_blk_tail; lane/arena.rs: the tp/tc scratch). */
Q8_API int q8_gemv(const q8_mat *W, q8_mode mode, const float *x, const q8_act *xq, int64_t rows, float *y, q8_ws *ws,
            q8_stream stream);

/* Dense int8-mode projections of 16 to 64 activation rows (a prefill chunk's, a batch's, or q8_gemv's with that many
 * rows) can run on the tensor cores — the grouped tensor-core product of the mixture with one group holding every row
 * — instead of the CUDA cores.  rows: -1 (automatic, the default): a call of one matrix of at least 2048 x 2048 takes
 * the tensor cores from 32 rows on, where they are measured faster (a prefill chunk's O projection); 0: the CUDA cores
 * always; 16 to 64: every call from that many rows on.  Process-wide; set it before the calls (and the decode model's
 * first step) it should affect. */
Q8_API int q8_set_tensor_core_rows(int rows);

/* The fewest rows an expert group of a chunk's int8-mode mixture (moe_gate_up, moe_down_combine over rows > 1) needs
 * to take the grouped tensor-core product instead of the CUDA-core kernels: 16 to 64, or 0 for the CUDA cores always.
 * The default is 32 (on this part 16-row groups are measured faster on the CUDA cores, 32-row groups even, 64-row
 * groups faster on the tensor cores).  Groups of more than 64 rows stay on the CUDA cores.  Process-wide; set it before the calls (and
 * the prefill chunks or batch steps) it should affect. */
Q8_API int q8_set_grouped_tensor_core_rows(int rows);

/* Whether prefill_chunk's causal attention runs on the tensor cores (1, the default) or the CUDA cores (0).  The
 * tensor-core form scales each tile of queries, keys, values and weights by a power of two, splits every f32 value
 * into two f16 parts and accumulates the three significant products in f32 (about 2^-22 relative per product); a
 * tile holding an infinity or a NaN cannot be split, and q8_model_check then reports Q8_EUNSUPPORTED.
 * Process-wide. */
Q8_API int q8_set_tensor_core_attention(int on);

/* The fewest sequences of a batch decode step (q8_model_desc.batch) whose attention runs in the streamed form: one
 * CTA per (split of 8 position chunks, key/value head, sequence) with a copy warp bringing its key and value rows
 * into a ring of shared-memory stages by bulk copies while eight warps fold each stage into a running softmax; the
 * splits of a (sequence, head) are folded in split order by the last to arrive.  Smaller batches keep the chunked form
 * (a CTA per 64 positions, folded in clusters of 8).  Both compute qwen_emit's attention (emit_qwen30b_generate);
 * their results differ only in summation order.  min_batch: 0 for never, else at least 2 (the default is 8).  Read
 * when a step is launched or captured.  Process-wide. */
Q8_API int q8_set_streamed_batch_attention(int min_batch);

/* Whether a one-sequence decode step in an int8 activation mode runs its layers as one persistent launch (1) or as six
 * launches a layer (0, the default).  The persistent launch keeps one CTA on every SM for the whole step (a
 * cooperative launch), separates a layer's stages (the norm and q/k/v, the attention, its fold, O, the norm and router,
 * gate-up, down-and-combine) by grid-wide barriers, and copies the weights and cache rows that do not depend on the
 * token into shared memory while the stage before them runs.  Its results equal the launch-per-stage step's up to the
 * summation order of the attention (qwen_emit docs, emit_qwen30b_generate: the same layer).  A model takes it when
 * its shapes fit (d and dff multiples of 128, d at most 4096, a CTA's share of the cache and of each stage's rows
 * within shared memory), its routers are Q8_0, it has no shared expert, and every block-scale array starts on a
 * 16-byte boundary; q8_model_persistent says whether it does.  Read when a step is launched or captured (a model's
 * first decode_step captures its graph).  Process-wide. */
Q8_API int q8_set_persistent_decode(int on);

/* Debug export of the int8 paths: the q8_gemv call (y as above) that also writes dots[r][o][b] = the exact int32 dot
 * of weight block (o, b) with activation block (r, b), from the same device code; dots is device int32
 * [rows][W.rows][W.cols/32].  The mode is Q8_INT8ACT, or Q8_INT8ACT2 when xq->lo is not NULL: dots is then
 * [2][rows][W.rows][W.cols/32], the words' dots followed by the low words' dots. */
Q8_API int q8_gemv_blockdots(const q8_mat *W, const q8_act *xq, int64_t rows, int32_t *dots, float *y, q8_ws *ws,
                      q8_stream stream);

/* q8_gemv without a workspace, for callers that cannot allocate device memory when they call it (code running inside
 * an allocator's callbacks, loops that forbid allocation after start-up, hosts whose device memory another runtime
 * has already handed out).  The pages have no counterpart: this is an addition for such callers.  Arguments and
 * results are those of q8_gemv.  Scratch (the quantized activation when xq is NULL, and the partial sums of a matrix
 * cut along k) comes from a fixed array of Q8_NOALLOC_SCRATCH_BYTES bytes and Q8_NOALLOC_COUNTERS counters that the
 * library holds on every device that loads it, until the process exits; a call that would need more returns
 * Q8_ENOSPACE and launches nothing.  The call allocates nothing and frees nothing.  After its arguments pass their
 * checks it clears the counters it will use (an asynchronous memset on `stream`) and then launches.  The first call on each device
 * looks up the array's device address (cudaGetSymbolAddress); make that first call before any stream capture.  Every
 * call on a device shares the one array: calls that overlap on the GPU (other streams, other threads) race and must
 * be ordered by the caller. */
#define Q8_NOALLOC_SCRATCH_BYTES (8u << 20)
#define Q8_NOALLOC_COUNTERS 65536u
Q8_API int q8_gemv_noalloc(const q8_mat *W, q8_mode mode, const float *x, const q8_act *xq, int64_t rows, float *y,
                           q8_stream stream);

/* ---- a5-a8: the sparse mixture ------------------------------------------------------------------------------------ */

/* Grouping of a chunk's choices by expert (lane_link.rs, Link::class_launch: MoeTokenSort; lane/arena.rs, scratch:
 * ec/eo/el): counts[e] choices of expert e, offsets[e] = sum of counts before e (offsets[experts] = rows*k), and
 * lists[offsets[e] .. offsets[e+1]) the choice indices r*k + j of expert e in ascending order.  Device int32 arrays. */
typedef struct {
    int32_t *counts;  /* [experts] */
    int32_t *offsets; /* [experts + 1] */
    int32_t *lists;   /* [rows * k] */
    int32_t *active;  /* [experts + 1]: the number of experts with choices, then those experts ascending */
} q8_moe_plan;

/* Router and top-k (forward_shim.rs, kernel_refusal Moe arms; lane_link.rs, Link::prim Moe: k <= 32, experts <= 8192):
 * l = router . x_r (the projection in `mode`), p = softmax(l), the k largest kept in descending order (equal logits:
 * lower expert first), g_j = p_j / sum of the kept p.  ids: device int32 [rows][k]; gates: device f32 [rows][k];
 * logits: device f32 [rows][experts] or NULL; plan: filled when not NULL.  experts = router->rows.  Several rows
 * spread over several CTAs; with a plan the last one to finish groups the choices, counted on one of the workspace's
 * arrival counters (left zero). */
Q8_API int moe_route_topk(const q8_mat *router, q8_mode mode, const float *x, const q8_act *xq, int64_t rows, int k,
                   int32_t *ids, float *gates, float *logits, const q8_moe_plan *plan, q8_ws *ws, q8_stream stream);

/* A shared expert (lane_link.rs, Link::class_launch: SharedExpertFusion, the mixture with the shared expert's gated
 * pair and down product in one launch; SharedExperts {wg, wu, wd, dff}): a SwiGLU feed-forward every row passes
 * through, its output added unweighted to the kept experts' weighted sum.  gate and up are [sdff, d], down [d, sdff]
 * (Q8_0, sdff % 32 == 0).  Where a call takes one, its hidden rows follow the routed ones in h (and hq): h is
 * [rows*k*dff + rows*sdff]. */
typedef struct {
    q8_mat gate, up, down;
} q8_shared_expert;

/* Router and top-k over a router of f32 values (lane_link.rs, Link::prim Moe: Router::F32, a router that is values
 * rather than quantized checkpoint rows): l = router . x_r with router device f32 [experts][d] (16-byte aligned,
 * d % 32 == 0) and x the f32 activation (in every mode: the router reads no quantized form), products summed in f32
 * per 128 values and then in f64; then top-k, gates and the grouping as moe_route_topk. */
Q8_API int moe_route_topk_f32(const float *router, int64_t experts, int64_t d, const float *x, int64_t rows, int k,
                              int32_t *ids, float *gates, float *logits, const q8_moe_plan *plan, q8_ws *ws,
                              q8_stream stream);

/* Gate-up with SwiGLU (qwen_emit, MoeWeights: gate/up [E*dff, d] stacked, expert e's rows at e*dff; emit_moe_forward:
 * each expert's SwiGLU at an expert-indexed base): h[r][j][i] = silu(Wg[e*dff+i] . x_r) * (Wu[e*dff+i] . x_r) with
 * e = ids[r][j], silu(z) = z/(1+e^-z).  h: device f32 [rows][k][dff].  In the int8 modes hq (device, words
 * [rows*k*dff] + scales [rows*k*dff/32], in Q8_INT8ACT2 with low words, or NULL) receives quantize(h)
 * (dff % 32 == 0); in the f32 mode it is ignored.
 * plan (from moe_route_topk) is required when rows > 1: each expert's weights are then read once for all its rows.
 * shared (or NULL): a shared expert whose hidden rows are written after the routed ones (one row: rows of the same
 * launch; a chunk: a projection of every row and a SwiGLU pass after the routed launches). */
Q8_API int moe_gate_up(const q8_mat *gate, const q8_mat *up, int64_t dff, q8_mode mode, const float *x, const q8_act *xq,
                int64_t rows, int k, const int32_t *ids, const q8_moe_plan *plan, float *h, const q8_act *hq,
                const q8_shared_expert *shared, q8_ws *ws, q8_stream stream);

/* Down-and-combine (qwen_emit, MoeWeights: down [E*d, dff] stacked, expert e's rows at e*d; emit_moe_forward: the
 * weighted combine): y[r] = residual[r] + sum_j gates[r][j] * (Wd[e*d .. e*d+d) . h[r][j]), the sum over j in order.
 * Mode Q8_F32ACT_F64SUM reads h; the int8 modes read hq (in Q8_INT8ACT2 with its low words), or quantize h when hq
 * is NULL.  residual may be NULL (and may alias y); y is device f32 [rows][d]; expert_out (device f32 [rows][k][d] or
 * NULL) receives each expert's unweighted output.  shared (or NULL): the shared expert of moe_gate_up, whose output is
 * added after the kept experts' (one row: blocks of the same launch; a chunk: a projection onto y after the combine). */
Q8_API int moe_down_combine(const q8_mat *down, int64_t d, q8_mode mode, const float *h, const q8_act *hq, int64_t rows,
                     int k, const int32_t *ids, const float *gates, const q8_moe_plan *plan, const float *residual,
                     float *y, float *expert_out, const q8_shared_expert *shared, q8_ws *ws, q8_stream stream);

/* ---- a10-a11: the decode step ----------------------------------------------------------------------------------- */

/* A model for decode_step (qwen_emit, emit_qwen30b_generate: RMSNorm -> Q/K/V -> per-head QK-norm + RoPE -> attention
 * over the KV cache -> O-proj -> residual -> RMSNorm -> mixture -> residual, per layer; then the LM head and the greedy
 * token).  Arrays named [layers] are HOST arrays of per-layer DEVICE pointers or matrices; q8_model_create copies
 * them.  Every device buffer stays owned by the caller and must outlive the model. */
typedef struct {
    int64_t layers, d, heads, kv_heads, head_dim, experts, k, dff, vocab, ctx;
    float eps;                  /* RMSNorm and QK-norm epsilon */
    double rope_theta;          /* RoPE base; pairs (i, i + head_dim/2) */
    q8_mode mode;
    const float *embed;         /* device f32 [vocab][d] */
    const float *const *attn_norm, *const *ffn_norm; /* [layers] -> device f32 [d] */
    const float *const *q_norm, *const *k_norm;      /* [layers] -> device f32 [head_dim] */
    const float *final_norm;    /* device f32 [d] */
    const q8_mat *wq, *wk, *wv, *wo;           /* [layers]: [heads*hd, d], [kv*hd, d], [kv*hd, d], [d, heads*hd] */
    const q8_mat *router, *gate, *up, *down;   /* [layers]: [E, d], [E*dff, d], [E*dff, d], [E*d, dff] */
    q8_mat lm_head;                            /* [vocab, d] */
    float *const *k_cache, *const *v_cache;    /* [layers] -> device f32 [kv_heads][ctx][head_dim], 32-byte aligned */
    int32_t *tok;               /* device int32 [1]: the token the step reads; the step writes the next token here */
    int32_t *pos;               /* device int32 [1]: the position the step writes; the step adds 1 */
    float *logits;              /* device f32 [vocab] or NULL */
    /* Optional variants of the mixture (NULL / 0 when absent): */
    const float *const *router_f32;  /* [layers] -> device f32 [E][d] routers of values used in place of `router` */
    const q8_mat *shared_gate, *shared_up, *shared_down;  /* [layers]: a shared expert, [shared_dff, d] x 2, [d, shared_dff] */
    int64_t shared_dff;
    /* The batch form (lane/mod.rs: Form / FormKind::Batch, batch_io): `batch` sequences (0 or 1: one) step together,
     * every weight read once for all of them.  Then tok and pos are device int32 [batch], logits [batch][vocab], and
     * each layer's cache holds the sequences' caches one after another: [batch][kv_heads][ctx][head_dim]. */
    int64_t batch;
} q8_model_desc;

typedef struct q8_model q8_model;

/* Checks the descriptor, allocates the model's activation buffers and workspace on the current device and builds the
 * RoPE table.  Refuses shapes the kernels do not run (head_dim != 128, heads % kv_heads, d % 32, ...). */
Q8_API int q8_model_create(const q8_model_desc *desc, q8_model **model);
Q8_API void q8_model_destroy(q8_model *model);

/* One token (one per sequence in the batch form): reads *tok and *pos on the device, writes the new key/value rows at
 * *pos, the logits (if requested) and the next token into *tok, and advances *pos.  In the batch form sequence b reads
 * tok[b] and pos[b] and attends its own cache; its norms, projections, routing and experts run as rows of one chunk
 * (each expert's weights read once for every sequence that chose it), and a bad position anywhere leaves every
 * sequence's token and position unchanged.  The first call on a model captures the whole step as one CUDA graph on a
 * private capture of `stream`; every call then replays it on `stream` (qwen_emit docs: one captured graph replayed per
 * token, position and token in device memory).  The first call must not be made while `stream` is capturing.  A step
 * whose *pos is outside [0, ctx) writes nothing and leaves *tok and *pos unchanged (the error is counted in the
 * model's device error word). */
Q8_API int decode_step(q8_model *model, q8_stream stream);
/* The same step as plain launches, without a graph (for tests and graph-capture by the caller). */
Q8_API int decode_step_launches(q8_model *model, q8_stream stream);
/* Debug export: decode_step_launches that also copies the residual stream into hidden (device f32 [layers + 1][d]; in
 * the batch form [layers + 1][batch][d]):
 * row 0 is the stream entering the first layer (the token's embedding row), row l + 1 the stream leaving layer l
 * (after its attention and mixture sums).  Per layer the step's results are those of decode_step; the copies are
 * ordinary stream operations between the launches.  For parity checks of each layer against a reference fed the same
 * input (emit_qwen30b_generate's per-layer order). */
Q8_API int decode_step_trace(q8_model *model, float *hidden, q8_stream stream);
/* A chunk of `rows` token rows through every layer (the prefill of a prompt chunk): tokens is device int32 [rows]; row
 * r takes position *pos + r.  Each layer: RMSNorm of the rows, the q/k/v projection of all rows, QK-norm, RoPE and the
 * key/value append of every row at its position, then each row's attention over rows 0 .. its position (causal), the O
 * projection onto the residual, RMSNorm, routing with the expert grouping, gate-up and down-and-combine of the chunk
 * (each chosen expert's weights read once for all its rows).  Then the last row's final norm, LM head and greedy token
 * into *tok; *pos advances by `rows`.  The result equals `rows` decode steps fed these tokens (up to the summation
 * order of the multi-row kernels).  The chunk's activations and every launch's scratch come from `ws` (Q8_ENOSPACE if
 * too small; about 0.7 MB a row at d 2048, 32 heads of 128 and a 4096-row cache); plain launches on `stream`, no
 * graph.  An id outside [0, vocab) or a row past the cache end sets the
 * model's device error word (q8_model_check).  Not for the batch form. */
Q8_API int prefill_chunk(q8_model *model, const int32_t *tokens, int64_t rows, q8_ws *ws, q8_stream stream);
/* prefill_chunk that also exports, for per-layer parity checks, the residual rows entering every layer and the final
 * ones (the input of the final norm): hidden is device f32 [layers + 1][rows][d]. */
Q8_API int prefill_chunk_trace(q8_model *model, const int32_t *tokens, int64_t rows, q8_ws *ws, float *hidden,
                               q8_stream stream);
/* Kernels one step launches: the kernel nodes of the graph the first decode_step captured (0 before it). */
Q8_API int64_t q8_model_launches_per_step(const q8_model *model);
/* 1 when the model's decode steps run their layers as one persistent launch (q8_set_persistent_decode), else 0. */
Q8_API int q8_model_persistent(const q8_model *model);
/* Reads and clears the model's device error word (synchronizes `stream`): Q8_OK, Q8_EINVAL when a step met an
 * out-of-range position or token, or Q8_ETIMEOUT when a bounded pipeline wait gave up. */
Q8_API int q8_model_check(q8_model *model, q8_stream stream);
/* Self-test of the bounded waits: one thread waits on a shared-memory barrier that nothing ever arrives on, giving up
 * after `polls` polls (1 to 2^20) exactly as the step's pipeline waits give up, and records the timeout in the model's
 * error word, which the next q8_model_check reports as Q8_ETIMEOUT.  Nothing else is touched. */
Q8_API int q8_model_wait_selftest(q8_model *model, unsigned polls, q8_stream stream);

/* ---- errors --------------------------------------------------------------------------------------------------- */
/* The text of the calling thread's last error (empty when none); valid until the thread's next call. */
Q8_API const char *q8_last_error(void);

#ifdef __cplusplus
}
#endif
#endif
