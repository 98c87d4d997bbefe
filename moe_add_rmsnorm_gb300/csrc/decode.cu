// The decode step's attention side and its last stage: single-query GQA attention split over positions, with the
// per-head QK-norm + RoPE and the KV append done inside it, and the greedy arg-max that advances token and position on
// the device.
//
// What it computes: qwen_emit docs, emit_qwen30b_generate (per-head QK-norm + RoPE, causal attention over a KV cache,
// device-side position and token); forward_shim.rs, kernel_refusal (Rope: a full rotary; Attention: scores scaled by
// 1/sqrt(HD), query heads grouped evenly over key/value heads, no mask, window, sink or soft cap) and
// ForwardShim::supports (KvCacheQuant refused: the caches are f32); lane_link.rs, Link::prim (Rope, Attention with its
// splits over positions, ArgMax) and Link::class_launch (FusedSampling: the arg-max advances token and position);
// lane/arena.rs, scratch (ap partials and ac counters of a split attention; av/ai/ac of the arg-max).
//
// How (GB300 design): the f32 cache is the second-largest byte stream of the step (one key and one value row of 512 B
// per position and key/value head), so the attention is a streaming kernel: every (key/value head, chunk of
// positions) pair is one CTA that reads its rows once with coalesced 16-byte loads and serves all query heads of its
// group from those registers; chunk partials (max, sum, weighted values) are folded in chunk order, first inside a
// thread-block cluster of 8 chunks through distributed shared memory, then across clusters by the last to arrive.  The
// 48 KiB static score row of the pages' design is not needed: a chunk's scores live in shared memory and any cache
// length works.  Every CTA norms and turns its group's query heads itself (a few hundred values), so no launch sits
// between the projection and the attention; the CTA whose chunk holds the new position also norms and turns the new
// key row and writes it and the value row to the caches.  Batches of many sequences attend in a streamed form instead
// (attention_stream_kernel): a CTA takes a long run of one sequence's positions and streams its rows through a ring of
// bulk copies with a running softmax, since the (sequence, head) pairs already fill the GPU.
#include <float.h>

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "stream.cuh"
#include "tcgen05.cuh"

namespace cg = cooperative_groups;

namespace q8 {
namespace {


// ==== attention ===================================================================================================

constexpr int ATT_THREADS = 256;
constexpr int ATT_CHUNK = 64;   // positions per CTA (8 per warp)
constexpr int ATT_MAXG = 8;     // query heads per key/value head
constexpr int ATT_HD = 128;     // head width the kernel is built for
constexpr int ATT_QP = 36;      // padded 32-dim quarter of a query row in shared memory: 16-byte reads, no conflicts
constexpr int ATT_CLUSTER = 8;  // chunks per thread-block cluster
constexpr int ATT_FOLD_B = 16;  // cluster partials a thread loads at once in the final fold

struct AttnParams {
    const float* q;        // the projection's q, k and v rows, before QK-norm and RoPE
    const float* k;
    const float* v;
    const float* q_norm;
    const float* k_norm;
    const float* cos_t;    // [ctx][ATT_HD / 2]
    const float* sin_t;
    float eps;
    int* err;
    float* k_cache;
    float* v_cache;
    const int32_t* pos;
    int heads, kv, ctx, G;
    float scale;
    float* out;
    int8_t* outq;
    int8_t* outl;  // with outq: the two-word form's low words
    float* outs;
    float* part;   // [kv][G][ncl_max][ATT_HD + 2]: each cluster's fold
    int* cnt;      // [kv * G]
    int nch_max;
    int ncl_max;
    int64_t cache_stride;  // batch form: the next sequence's caches (its q/k/v/out rows, position, scratch follow theirs)
    L2Prefetch pf;
};

// The batch form's sequence b (blockIdx.z): its rows, caches, position, outputs and fold scratch.
__device__ __forceinline__ AttnParams attn_for_sequence(const AttnParams& p0, int b) {
    AttnParams p = p0;
    const int64_t qd = (int64_t)p0.heads * ATT_HD, kd = (int64_t)p0.kv * ATT_HD;
    p.q += b * qd;
    p.k += b * kd;
    p.v += b * kd;
    p.k_cache += b * p0.cache_stride;
    p.v_cache += b * p0.cache_stride;
    p.pos += b;
    p.out += b * qd;
    if (p.outq) p.outq += b * qd;
    if (p.outl) p.outl += b * qd;
    if (p.outs) p.outs += b * qd / 32;
    p.part += (int64_t)b * p0.heads * p0.ncl_max * (ATT_HD + 2);
    p.cnt += (int64_t)b * p0.heads;
    return p;
}

// A chunk's partial: per query head its weighted values (ATT_HD), its max score and its sum of exponentials.
__shared__ __align__(16) float att_partial[ATT_MAXG][ATT_HD + 2];

// The cluster's chunks are folded by rank: CTA rank r takes query heads r, r + 4, ... of the group and reads each
// head's partial from every CTA of the cluster through distributed shared memory, in rank order.  The cluster's result goes to global scratch; the
// last cluster of the key/value head to arrive (per query head) folds the clusters' results in cluster order, writes
// the head's output and quantizes it.  Fold: M = max m_c, out = sum exp(m_c - M) acc_c / sum exp(m_c - M) l_c.
__device__ void fold_cluster(const AttnParams& p, int g, int chunk, int G, int t) {
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ int last[ATT_MAXG];
    __shared__ float fm[ATT_MAXG][ATT_CLUSTER];
    cluster.sync();  // every chunk's partial is in its CTA's shared memory
    const int rank = (int)cluster.block_rank();
    const int cl = chunk / ATT_CLUSTER;
    const int ncl = p.ncl_max;
    // this rank's query heads: rank, rank + ATT_CLUSTER, ...
    for (int hh = rank; hh < G; hh += ATT_CLUSTER)
        if (t < ATT_CLUSTER) fm[hh][t] = cluster.map_shared_rank(&att_partial[0][0], t)[hh * (ATT_HD + 2) + ATT_HD];
    __syncthreads();
    for (int hh = rank; hh < G; hh += ATT_CLUSTER) {
        float* out_part = p.part + (((int64_t)g * G + hh) * ncl + cl) * (ATT_HD + 2);
        float M = -FLT_MAX;
#pragma unroll
        for (int c = 0; c < ATT_CLUSTER; ++c) M = fmaxf(M, fm[hh][c]);
        if (t < ATT_HD + 2) {
            const int col = (t == ATT_HD) ? ATT_HD + 1 : t;  // thread ATT_HD folds the sums; ATT_HD+1 writes M
            float acc = 0.f;
            if (t != ATT_HD + 1)
#pragma unroll
                for (int c = 0; c < ATT_CLUSTER; ++c) {
                    const float* src = cluster.map_shared_rank(&att_partial[0][0], c) + hh * (ATT_HD + 2);
                    const float f = fm[hh][c] == -FLT_MAX ? 0.f : expf(fm[hh][c] - M);
                    acc = fmaf(f, src[col], acc);
                }
            if (t < ATT_HD) out_part[t] = acc;
            else if (t == ATT_HD) out_part[ATT_HD + 1] = acc;
            else out_part[ATT_HD] = M;
        }
    }
    cluster_arrive();  // this CTA has read the others' partials; it waits for theirs only before it exits
    if (rank >= G) {
        cluster_wait();
        return;
    }
    __syncthreads();  // the CTA's cluster results are written
    const int ncl_used = (((*p.pos + 1) + ATT_CHUNK - 1) / ATT_CHUNK + ATT_CLUSTER - 1) / ATT_CLUSTER;
    if (t < ATT_MAXG) {  // the arrival releases them (cumulative over the barrier) and acquires the others'
        const int hh = rank + t * ATT_CLUSTER;
        last[t] = hh < G ? (atomic_add_acq_rel_gpu(p.cnt + g * G + hh, 1) == ncl_used - 1) : 0;
    }
    __syncthreads();  // the other threads read after the arriving thread's acquire
    // the heads this CTA arrived last for (rank, and rank + ATT_CLUSTER when a group has more heads than the cluster
    // has CTAs) are folded at once, 128 threads a head,
    // thread d summing dimension d over the clusters
    const int lane = t & 31;
    const int u = t / ATT_HD, d = t % ATT_HD;  // head slot, dimension
    const int hh = rank + u * ATT_CLUSTER;
    const bool mine = hh < G && last[u];       // uniform over the slot's four warps
    const bool any = last[0] || (ATT_CLUSTER < G && last[1]);
    if (!any) {
        cluster_wait();
        return;
    }
    const float* base = p.part + ((int64_t)g * G + (mine ? hh : 0)) * ncl * (ATT_HD + 2);
    if (mine) {
        // batches of 16 clusters, all loads of a batch in flight; the running maximum rescales the sums (online
        // softmax), so no separate pass finds the maximum first
        float M = -FLT_MAX, num = 0.f, den = 0.f;
        for (int cb = 0; cb < ncl_used; cb += ATT_FOLD_B) {
            float mc[ATT_FOLD_B], vc[ATT_FOLD_B], lc[ATT_FOLD_B];
#pragma unroll
            for (int i = 0; i < ATT_FOLD_B; ++i) {
                const int c = cb + i;
                const float* b = base + (int64_t)(c < ncl_used ? c : ncl_used - 1) * (ATT_HD + 2);
                mc[i] = c < ncl_used ? __ldcg(b + ATT_HD) : -FLT_MAX;
                vc[i] = c < ncl_used ? __ldcg(b + d) : 0.f;
                lc[i] = c < ncl_used ? __ldcg(b + ATT_HD + 1) : 0.f;
            }
            float Mb = M;
#pragma unroll
            for (int i = 0; i < ATT_FOLD_B; ++i) Mb = fmaxf(Mb, mc[i]);
            if (Mb != -FLT_MAX) {
                const float r = M == -FLT_MAX ? 0.f : expf(M - Mb);
                num *= r;
                den *= r;
#pragma unroll
                for (int i = 0; i < ATT_FOLD_B; ++i) {
                    const float f = mc[i] == -FLT_MAX ? 0.f : expf(mc[i] - Mb);
                    num = fmaf(f, vc[i], num);
                    den = fmaf(f, lc[i], den);
                }
                M = Mb;
            }
        }
        const float o = num / den;
        const int64_t oi = ((int64_t)g * G + hh) * ATT_HD + d;
        p.out[oi] = o;
        if (p.outq) {  // the slot's four warps hold the head's four 32-value blocks
            float dsc;
            if (p.outl) {
                int8_t lv;
                p.outq[oi] = quantize2_lane(o, dsc, lv);
                p.outl[oi] = lv;
            } else {
                p.outq[oi] = quantize_lane(o, dsc);
            }
            if (lane == 0) p.outs[oi / 32] = dsc;
        }
        if (d == 0) p.cnt[g * G + hh] = 0;
    }
    cluster_wait();  // no CTA leaves while another may still read its shared memory
}

// grid (kv, chunk) in clusters of 8 chunks, 8 warps, two CTAs per SM.  Scores: 4 lanes per position (a 32-dim quarter
// each), each warp 8 positions.  Values: warp w takes positions w, w+8, ... (8 rows), lane l the dims 4l..4l+3; every
// key and value row is loaded before any is used; the 8 warps' sums meet in shared memory.  A chunk's partial
// is then folded with the rest of its cluster and across clusters (fold_cluster), always in chunk order.
template <bool BATCH>
__global__ void __launch_bounds__(ATT_THREADS, 2) attention_kernel(const AttnParams pk) {
    const AttnParams p = BATCH ? attn_for_sequence(pk, blockIdx.z) : pk;
    __shared__ __align__(16) float qs[ATT_MAXG][4 * ATT_QP];
    __shared__ __align__(16) float sc[ATT_MAXG][ATT_CHUNK];
    __shared__ __align__(16) float red[ATT_THREADS / 32][ATT_MAXG][ATT_HD];  // [warp][g][dim]; float4 stores
    __shared__ float stat[ATT_MAXG][2];
    __shared__ __align__(16) float knew[ATT_HD];
    __shared__ __align__(16) float vnew[ATT_HD];
    __shared__ float nred[ATT_MAXG + 1][2];
    const int g = blockIdx.x, chunk = blockIdx.y;
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int G = p.G;
    issue_l2_prefetch(p.pf);
    // The position is fixed for the whole step (the previous step's last kernel wrote it), and every cached row but
    // the new one at `pos` was written by earlier steps: those rows are read before waiting for the kernels of this
    // step; the new row and the queries after.
    const int len = *p.pos + 1;  // rows 0..pos
    const int nch = (len + ATT_CHUNK - 1) / ATT_CHUNK;
    // a whole cluster past the cache end (or a bad position) leaves together; a chunk past the end inside a working
    // cluster contributes an empty partial
    if (len < 1 || len > p.ctx || (chunk / ATT_CLUSTER) * ATT_CLUSTER >= nch) {
        griddep_wait();
        griddep_launch();
        if ((len < 1 || len > p.ctx) && g == 0 && chunk == 0 && t == 0 && p.err) atomicOr(p.err, 2);
        return;
    }
    // QK-norm and RoPE constants for this position, read first (before the bulk of the cache rows): thread t takes
    // the pair (i, i + 64) of query heads t/64 and t/64 + 4 (and of the key head when t < 64)
    const int hsub = t >> 6, pi = t & 63;
    const int pos = len - 1;
    const float cs = ld_f32_early(p.cos_t + (int64_t)pos * (ATT_HD / 2) + pi);
    const float sn = ld_f32_early(p.sin_t + (int64_t)pos * (ATT_HD / 2) + pi);
    const float qw0 = ld_f32_early(p.q_norm + pi), qw1 = ld_f32_early(p.q_norm + pi + ATT_HD / 2);
    const float kw0 = ld_f32_early(p.k_norm + pi), kw1 = ld_f32_early(p.k_norm + pi + ATT_HD / 2);
    const int p0 = chunk * ATT_CHUNK;
    const int np = max(0, min(ATT_CHUNK, len - p0));
    const int newrow = len - 1 - p0;  // the row this step writes, if it falls in this chunk
    const float* kb = p.k_cache + ((int64_t)g * p.ctx + p0) * ATT_HD;
    const float* vb = p.v_cache + ((int64_t)g * p.ctx + p0) * ATT_HD;
    const int sub = lane & 3;
    constexpr int PASSES = ATT_CHUNK / 64;
    float kr[PASSES][32];
    float4 vr[ATT_CHUNK / 8];
#pragma unroll
    for (int pass = 0; pass < PASSES; ++pass) {
        const int pl = pass * 64 + wid * 8 + (lane >> 2);
        const bool pre = pl < np && pl != newrow;
        const float* kp = kb + (int64_t)(pre ? pl : 0) * ATT_HD + sub * 32;
        // four 32-byte loads: each instruction reads whole sectors (lane quarter = 128 contiguous bytes)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (pre) {
                ld_f8_stream(kp + 8 * i, &kr[pass][8 * i]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) kr[pass][8 * i + e] = 0.f;
            }
        }
    }
#pragma unroll
    for (int u = 0; u < ATT_CHUNK / 8; ++u) {
        const int pl = wid + 8 * u;
        vr[u] = (pl < np && pl != newrow) ? __ldcs(reinterpret_cast<const float4*>(vb + (int64_t)pl * ATT_HD) + lane)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const bool has_new = newrow >= 0 && newrow < np;  // CTA-uniform
    griddep_wait();
    griddep_launch();
    // the projection's rows of this step: the group's queries, and the key and value rows the new position appends
    float qa[2], qb[2], ka = 0.f, kb2 = 0.f, va = 0.f, vb2 = 0.f;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int hh = hsub + 4 * u;
        const float* src = p.q + ((int64_t)g * G + (hh < G ? hh : 0)) * ATT_HD;
        qa[u] = hh < G ? __ldcg(src + pi) : 0.f;
        qb[u] = hh < G ? __ldcg(src + pi + ATT_HD / 2) : 0.f;
    }
    if (has_new && t < 64) {
        ka = __ldcg(p.k + (int64_t)g * ATT_HD + pi);
        kb2 = __ldcg(p.k + (int64_t)g * ATT_HD + pi + ATT_HD / 2);
    } else if (has_new && t < 128) {
        va = __ldcg(p.v + (int64_t)g * ATT_HD + pi);
        vb2 = __ldcg(p.v + (int64_t)g * ATT_HD + pi + ATT_HD / 2);
    }
    // per-head sum of squares: a head's 64 threads are two warps
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const float ss = group_sum<32>(qa[u] * qa[u] + qb[u] * qb[u]);
        if (lane == 0) nred[hsub + 4 * u][wid & 1] = ss;
    }
    {
        const float ss = group_sum<32>(ka * ka + kb2 * kb2);
        if (lane == 0 && t < 64) nred[ATT_MAXG][wid & 1] = ss;
    }
    __syncthreads();
    // per-head RMSNorm (eps inside the root, the head weight multiplies), then the NeoX rotation of (i, i + 64)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int hh = hsub + 4 * u;
        if (hh < G) {
            const float tot = (0.f + nred[hh][0]) + nred[hh][1];
            const float inv = 1.0f / sqrtf(tot / (float)ATT_HD + p.eps);
            const float a = qa[u] * inv * qw0, b = qb[u] * inv * qw1;
            const float ra = a * cs - b * sn, rb = a * sn + b * cs;
            qs[hh][(pi >> 5) * ATT_QP + (pi & 31)] = ra;
            qs[hh][((pi + 64) >> 5) * ATT_QP + (pi & 31)] = rb;
        }
    }
    if (has_new) {
        if (t < 64) {
            const float tot = (0.f + nred[ATT_MAXG][0]) + nred[ATT_MAXG][1];
            const float inv = 1.0f / sqrtf(tot / (float)ATT_HD + p.eps);
            const float a = ka * inv * kw0, b = kb2 * inv * kw1;
            const float ra = a * cs - b * sn, rb = a * sn + b * cs;
            knew[pi] = ra;
            knew[pi + ATT_HD / 2] = rb;
            float* kr_out = p.k_cache + ((int64_t)g * p.ctx + pos) * ATT_HD;
            kr_out[pi] = ra;
            kr_out[pi + ATT_HD / 2] = rb;
        } else if (t < 128) {
            vnew[pi] = va;
            vnew[pi + ATT_HD / 2] = vb2;
            float* vr_out = p.v_cache + ((int64_t)g * p.ctx + pos) * ATT_HD;
            vr_out[pi] = va;
            vr_out[pi + ATT_HD / 2] = vb2;
        }
    }
    __syncthreads();
    if (has_new) {  // the lanes that hold the new row take it from shared memory
#pragma unroll
        for (int pass = 0; pass < PASSES; ++pass) {
            const int pl = pass * 64 + wid * 8 + (lane >> 2);
            if (pl == newrow) {
                const float4* kp = reinterpret_cast<const float4*>(knew + sub * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 v = kp[i];
                    kr[pass][4 * i] = v.x;
                    kr[pass][4 * i + 1] = v.y;
                    kr[pass][4 * i + 2] = v.z;
                    kr[pass][4 * i + 3] = v.w;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < ATT_CHUNK / 8; ++u)
            if (wid + 8 * u == newrow) vr[u] = reinterpret_cast<const float4*>(vnew)[lane];
    }
    // scores (every lane runs the same path; lanes past the chunk's end multiply zeros and store nothing)
#pragma unroll
    for (int pass = 0; pass < PASSES; ++pass) {
        const int pl = pass * 64 + wid * 8 + (lane >> 2);
        const bool valid = pl < np;
        for (int hh = 0; hh < G; ++hh) {
            const float4* qv = reinterpret_cast<const float4*>(&qs[hh][sub * ATT_QP]);
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 q4 = qv[i];
                acc = fmaf(q4.x, kr[pass][4 * i], acc);
                acc = fmaf(q4.y, kr[pass][4 * i + 1], acc);
                acc = fmaf(q4.z, kr[pass][4 * i + 2], acc);
                acc = fmaf(q4.w, kr[pass][4 * i + 3], acc);
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (sub == 0 && valid) sc[hh][pl] = acc * p.scale;
        }
    }
    __syncthreads();
    // chunk softmax statistics per head (warp hh), scores replaced by exp(s - m)
    for (int hh = wid; hh < G; hh += ATT_THREADS / 32) {
        float m = -FLT_MAX;
        for (int i = lane; i < np; i += 32) m = fmaxf(m, sc[hh][i]);
        m = warp_max(m);
        float l = 0.f;
        for (int i = lane; i < np; i += 32) {
            const float e = expf(sc[hh][i] - m);
            sc[hh][i] = e;
            l += e;
        }
        l = group_sum<32>(l);
        if (lane == 0) {
            stat[hh][0] = np > 0 ? m : -FLT_MAX;
            stat[hh][1] = l;
        }
    }
    __syncthreads();
    // weighted values: the warp's 16 rows, already in registers
    {
#pragma unroll
        for (int hh = 0; hh < ATT_MAXG; ++hh) {
            if (hh < G) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int u = 0; u < ATT_CHUNK / 8; ++u) {
                    const int pl = wid + 8 * u;
                    const float w = pl < np ? sc[hh][pl] : 0.f;
                    acc.x = fmaf(w, vr[u].x, acc.x);
                    acc.y = fmaf(w, vr[u].y, acc.y);
                    acc.z = fmaf(w, vr[u].z, acc.z);
                    acc.w = fmaf(w, vr[u].w, acc.w);
                }
                *reinterpret_cast<float4*>(&red[wid][hh][4 * lane]) = acc;
            }
        }
    }
    __syncthreads();
    // this chunk's partial stays in shared memory for the cluster's fold
    for (int i = t; i < G * ATT_HD; i += ATT_THREADS) {
        const int hh = i / ATT_HD, dd = i % ATT_HD;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < ATT_THREADS / 32; ++w) s += red[w][hh][dd];
        att_partial[hh][dd] = s;
    }
    if (t < G) {
        att_partial[t][ATT_HD] = stat[t][0];
        att_partial[t][ATT_HD + 1] = stat[t][1];
    }
    fold_cluster(p, g, chunk, G, t);
}

// ==== the batch form's streamed attention ========================================================================
// Many sequences, each one query row against its own cache: the (sequence, key/value head) pairs already fill the GPU,
// so a CTA takes a long run of positions instead of one chunk and keeps the copy engine busy on it: one lane of the
// copy warp brings each stage of AS_SUB positions (its key rows, then its value rows: two contiguous bulk copies) into
// a ring of AS_STAGES stages while the eight compute warps work on an earlier one with a running (online) softmax.  The
// splits of a (sequence, key/value head) meet through global scratch: the last to arrive folds them in split order.

constexpr int AS_CW = 8;                      // compute warps
constexpr int AS_THREADS = (AS_CW + 1) * 32;  // + the copy warp
constexpr int AS_SUB = 32;                    // positions per stage
constexpr int AS_STAGES = 3;                  // (two CTAs an SM: one's start and end overlap the other's stream)
constexpr int AS_PPW = AS_SUB / AS_CW;        // positions a warp takes in a stage
constexpr int AS_LP = 32 / AS_PPW;            // lanes a position's score takes
constexpr int AS_FL = ATT_HD / 4 / AS_LP;     // float4 of the key row a lane takes
static_assert(AS_PPW % 4 == 0 && AS_LP <= 8, "whole float4 of weights; 8 lanes at most per position");
constexpr size_t AS_STAGE = 2 * (size_t)AS_SUB * ATT_HD * sizeof(float);  // keys, then values
constexpr size_t AS_SMEM = AS_STAGES * AS_STAGE;
static_assert(2 * (AS_SMEM + 12 * 1024) <= 232448, "two CTAs' rings and static arrays within an SM's shared memory");
static_assert((size_t)AS_CW * ATT_MAXG * ATT_HD * sizeof(float) <= AS_STAGE, "the warps' sums fit in a stage");

// grid (split, key/value head, sequence).  Split j of S takes the stages [j * nch / S, (j+1) * nch / S) of its
// sequence's nch = ceil(len / AS_SUB).  Scores: AS_LP lanes a position, lane s of them the float4 s, s + AS_LP, ... of
// the key row (with 4 lanes a position rotated by the position's parity), so that the 8 lanes of a shared-memory phase
// read 8 different bank groups; a warp AS_PPW positions.  Values: warp w takes positions AS_PPW w .., lane l the
// dimensions 4l..4l+3, the running sums rescaled by each stage's change of the running maximum.
__global__ void __launch_bounds__(AS_THREADS, 2) attention_stream_kernel(const AttnParams pk) {
    extern __shared__ __align__(128) unsigned char as_ring[];
    __shared__ __align__(16) float qs[ATT_MAXG][ATT_HD];
    __shared__ __align__(16) float sc[2][ATT_MAXG][AS_SUB];
    __shared__ float rfac[2][ATT_MAXG];
    __shared__ float run_m[ATT_MAXG], run_l[ATT_MAXG];
    __shared__ __align__(16) float knew[ATT_HD];
    __shared__ __align__(16) float vnew[ATT_HD];
    __shared__ float nred[ATT_MAXG + 1][2];
    __shared__ __align__(8) uint64_t full[AS_STAGES], empty[AS_STAGES];
    __shared__ int last_s;
    const AttnParams p = attn_for_sequence(pk, blockIdx.z);
    const int split = blockIdx.x, S = gridDim.x, g = blockIdx.y;
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int G = p.G;
    const int len = *p.pos + 1;
    if (len < 1 || len > p.ctx) {  // a bad position: nothing is read or written
        griddep_wait();
        griddep_launch();
        if (split == 0 && g == 0 && t == 0 && p.err) atomicOr(p.err, 2);
        return;
    }
    const int nch = (len + AS_SUB - 1) / AS_SUB;
    const int c0 = split * nch / S, nst = (split + 1) * nch / S - c0;
    const int pos = len - 1;
    const bool has_new = nst > 0 && c0 + nst == nch;  // this split holds the last stage, whose last row is new
    if (t == 0) {
        for (int i = 0; i < AS_STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], AS_CW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    const float* kb = p.k_cache + (int64_t)g * p.ctx * ATT_HD;
    const float* vb = p.v_cache + (int64_t)g * p.ctx * ATT_HD;
    if (wid == AS_CW) {
        // ---- the copy warp: stage i = positions AS_SUB (c0 + i) .. of the cached rows (the new row is not read) ----
        // The cached rows were written by earlier steps, so the first stages go out before the wait for this step's
        // kernels.
        if (lane == 0) {
            bool ok = true;
            int issued = 0;
            for (int i = 0; i < nst && ok; ++i, ++issued) {
                const int slot = i % AS_STAGES;
                if (i >= AS_STAGES) ok = mbar_wait(&empty[slot], ((i / AS_STAGES) - 1) & 1, p.err);
                if (!ok) break;
                const int p0 = (c0 + i) * AS_SUB;
                int rows = min(AS_SUB, len - p0);
                if (c0 + i == nch - 1) --rows;  // the new position is the last row
                unsigned char* st = as_ring + (size_t)slot * AS_STAGE;
                const unsigned rb = (unsigned)rows * ATT_HD * sizeof(float);
                mbar_arrive_expect_tx(&full[slot], 2u * rb);
                if (rows > 0) {
                    bulk_g2s(st, kb + (int64_t)p0 * ATT_HD, rb, &full[slot]);
                    bulk_g2s(st + AS_STAGE / 2, vb + (int64_t)p0 * ATT_HD, rb, &full[slot]);
                }
            }
            // every copy issued has landed before the CTA may end, after a timed-out wait too (each wait bounded)
            for (int i = max(0, issued - AS_STAGES); i < issued; ++i)
                mbar_wait(&full[i % AS_STAGES], (i / AS_STAGES) & 1, p.err);
        }
        griddep_wait();
        griddep_launch();
        __syncwarp();
    } else {
        griddep_wait();
        griddep_launch();
        // ---- QK-norm and RoPE of the group's queries (and of the new key row, in the split that holds it) ----------
        // thread t (< 256) takes the pair (i, i + 64) of query heads t/64 and t/64 + 4, and of the key head when t < 64
        const int hsub = t >> 6, pi = t & 63;
        const float cs = __ldg(p.cos_t + (int64_t)pos * (ATT_HD / 2) + pi);
        const float sn = __ldg(p.sin_t + (int64_t)pos * (ATT_HD / 2) + pi);
        float qa[2], qb[2], ka = 0.f, kb2 = 0.f, va = 0.f, vb2 = 0.f;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int hh = hsub + 4 * u;
            const float* src = p.q + ((int64_t)g * G + (hh < G ? hh : 0)) * ATT_HD;
            qa[u] = hh < G ? __ldcg(src + pi) : 0.f;
            qb[u] = hh < G ? __ldcg(src + pi + ATT_HD / 2) : 0.f;
        }
        if (has_new && t < 64) {
            ka = __ldcg(p.k + (int64_t)g * ATT_HD + pi);
            kb2 = __ldcg(p.k + (int64_t)g * ATT_HD + pi + ATT_HD / 2);
        } else if (has_new && t < 128) {
            va = __ldcg(p.v + (int64_t)g * ATT_HD + pi);
            vb2 = __ldcg(p.v + (int64_t)g * ATT_HD + pi + ATT_HD / 2);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const float ss = group_sum<32>(qa[u] * qa[u] + qb[u] * qb[u]);
            if (lane == 0) nred[hsub + 4 * u][wid & 1] = ss;
        }
        {
            const float ss = group_sum<32>(ka * ka + kb2 * kb2);
            if (lane == 0 && t < 64) nred[ATT_MAXG][wid & 1] = ss;
        }
        if (t < ATT_MAXG) {
            run_m[t] = -FLT_MAX;
            run_l[t] = 0.f;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(AS_CW * 32));
        const float qw0 = __ldg(p.q_norm + pi), qw1 = __ldg(p.q_norm + pi + ATT_HD / 2);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int hh = hsub + 4 * u;
            if (hh < G) {
                const float tot = (0.f + nred[hh][0]) + nred[hh][1];
                const float inv = 1.0f / sqrtf(tot / (float)ATT_HD + p.eps);
                const float a = qa[u] * inv * qw0, b = qb[u] * inv * qw1;
                qs[hh][pi] = a * cs - b * sn;
                qs[hh][pi + ATT_HD / 2] = a * sn + b * cs;
            }
        }
        if (has_new) {
            if (t < 64) {
                const float kw0 = __ldg(p.k_norm + pi), kw1 = __ldg(p.k_norm + pi + ATT_HD / 2);
                const float tot = (0.f + nred[ATT_MAXG][0]) + nred[ATT_MAXG][1];
                const float inv = 1.0f / sqrtf(tot / (float)ATT_HD + p.eps);
                const float a = ka * inv * kw0, b = kb2 * inv * kw1;
                const float ra = a * cs - b * sn, rb = a * sn + b * cs;
                knew[pi] = ra;
                knew[pi + ATT_HD / 2] = rb;
                float* kr_out = p.k_cache + ((int64_t)g * p.ctx + pos) * ATT_HD;
                kr_out[pi] = ra;
                kr_out[pi + ATT_HD / 2] = rb;
            } else if (t < 128) {
                vnew[pi] = va;
                vnew[pi + ATT_HD / 2] = vb2;
                float* vr_out = p.v_cache + ((int64_t)g * p.ctx + pos) * ATT_HD;
                vr_out[pi] = va;
                vr_out[pi + ATT_HD / 2] = vb2;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(AS_CW * 32));
        // ---- the stages -----------------------------------------------------------------------------------------------
        float4 acc[ATT_MAXG];
#pragma unroll
        for (int hh = 0; hh < ATT_MAXG; ++hh) acc[hh] = make_float4(0.f, 0.f, 0.f, 0.f);
        bool ok = true;
        const int sub = lane & (AS_LP - 1);
        for (int i = 0; i < nst; ++i) {
            const int slot = i % AS_STAGES, b = i & 1;
            if (ok) ok = mbar_wait(&full[slot], (i / AS_STAGES) & 1, p.err);
            float* K = reinterpret_cast<float*>(as_ring + (size_t)slot * AS_STAGE);
            float* V = K + AS_SUB * ATT_HD;
            const int p0 = (c0 + i) * AS_SUB;
            const int np = min(AS_SUB, len - p0);
            if (c0 + i == nch - 1) {  // the new row, from this CTA's own norm and rotation
                if (t < ATT_HD) K[(np - 1) * ATT_HD + t] = knew[t];
                else V[(np - 1) * ATT_HD + t - ATT_HD] = vnew[t - ATT_HD];
                asm volatile("bar.sync 1, %0;" ::"n"(AS_CW * 32));
            }
            // scores
            {
                const int pl = wid * AS_PPW + lane / AS_LP;
                const int rot = AS_LP < 8 ? AS_LP * (pl & 1) : 0;
                float4 k4[AS_FL];
                const float4* kr = reinterpret_cast<const float4*>(K + pl * ATT_HD);
#pragma unroll
                for (int j = 0; j < AS_FL; ++j) k4[j] = kr[(AS_LP * j + sub + rot) & 31];
                // every head's partial dot first, then their lane sums side by side (independent chains)
                float a[ATT_MAXG];
#pragma unroll
                for (int hh = 0; hh < ATT_MAXG; ++hh) {
                    a[hh] = 0.f;
                    if (hh < G) {  // uniform
                        const float4* qv = reinterpret_cast<const float4*>(qs[hh]);
#pragma unroll
                        for (int j = 0; j < AS_FL; ++j) {
                            const float4 q4 = qv[(AS_LP * j + sub + rot) & 31];
                            a[hh] = fmaf(q4.x, k4[j].x, a[hh]);
                            a[hh] = fmaf(q4.y, k4[j].y, a[hh]);
                            a[hh] = fmaf(q4.z, k4[j].z, a[hh]);
                            a[hh] = fmaf(q4.w, k4[j].w, a[hh]);
                        }
                    }
                }
#pragma unroll
                for (int o = 1; o < AS_LP; o <<= 1)
#pragma unroll
                    for (int hh = 0; hh < ATT_MAXG; ++hh) a[hh] += __shfl_xor_sync(0xffffffffu, a[hh], o);
                if (sub == 0 && pl < np)
#pragma unroll
                    for (int hh = 0; hh < ATT_MAXG; ++hh)
                        if (hh < G) sc[b][hh][pl] = a[hh] * p.scale;
            }
            asm volatile("bar.sync 1, %0;" ::"n"(AS_CW * 32));
            // the running softmax: warp hh takes head hh
            if (wid < G) {
                float m = -FLT_MAX;
                for (int r = lane; r < np; r += 32) m = fmaxf(m, sc[b][wid][r]);
                m = warp_max(m);
                const float mo = run_m[wid];
                const float mn = fmaxf(mo, m);
                float l = 0.f;
                for (int r = lane; r < np; r += 32) {
                    const float e = expf(sc[b][wid][r] - mn);
                    sc[b][wid][r] = e;
                    l += e;
                }
                l = group_sum<32>(l);
                if (lane == 0) {
                    const float f = mo == -FLT_MAX ? 0.f : expf(mo - mn);
                    rfac[b][wid] = f;
                    run_l[wid] = run_l[wid] * f + l;
                    run_m[wid] = mn;
                }
            }
            asm volatile("bar.sync 1, %0;" ::"n"(AS_CW * 32));
            // weighted values: warp w takes the consecutive positions AS_PPW w .., so a head's weights are whole float4
            {
                constexpr int PW = AS_PPW;
                float4 v4[PW];
#pragma unroll
                for (int u = 0; u < PW; ++u) {
                    const int pl = PW * wid + u;
                    v4[u] = pl < np ? reinterpret_cast<const float4*>(V + pl * ATT_HD)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int hh = 0; hh < ATT_MAXG; ++hh) {
                    if (hh < G) {
                        const float f = rfac[b][hh];
                        float4 a = make_float4(acc[hh].x * f, acc[hh].y * f, acc[hh].z * f, acc[hh].w * f);
                        float wv[PW];
#pragma unroll
                        for (int f4 = 0; f4 < PW / 4; ++f4) {
                            const float4 w4 = *reinterpret_cast<const float4*>(&sc[b][hh][PW * wid + 4 * f4]);
                            wv[4 * f4] = w4.x;
                            wv[4 * f4 + 1] = w4.y;
                            wv[4 * f4 + 2] = w4.z;
                            wv[4 * f4 + 3] = w4.w;
                        }
#pragma unroll
                        for (int u = 0; u < PW; ++u) {
                            const int pl = PW * wid + u;
                            if (pl < np) {  // warp-uniform (a weight past np was never written)
                                const float w = wv[u];
                                a.x = fmaf(w, v4[u].x, a.x);
                                a.y = fmaf(w, v4[u].y, a.y);
                                a.z = fmaf(w, v4[u].z, a.z);
                                a.w = fmaf(w, v4[u].w, a.w);
                            }
                        }
                        acc[hh] = a;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        // ---- this split's partial: the warps' sums meet in the first stage of the ring (every copy has been used) ----
        asm volatile("bar.sync 1, %0;" ::"n"(AS_CW * 32));
        float* red = reinterpret_cast<float*>(as_ring);  // [warp][head][dim]
#pragma unroll
        for (int hh = 0; hh < ATT_MAXG; ++hh)
            if (hh < G) *reinterpret_cast<float4*>(red + ((size_t)wid * ATT_MAXG + hh) * ATT_HD + 4 * lane) = acc[hh];
        asm volatile("bar.sync 1, %0;" ::"n"(AS_CW * 32));
        const int ncl = p.ncl_max;
        for (int i = t; i < G * ATT_HD; i += AS_CW * 32) {
            const int hh = i / ATT_HD, dd = i % ATT_HD;
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < AS_CW; ++w) s += red[((size_t)w * ATT_MAXG + hh) * ATT_HD + dd];
            p.part[(((int64_t)g * G + hh) * ncl + split) * (ATT_HD + 2) + dd] = s;
        }
        if (t < G) {
            float* o = p.part + (((int64_t)g * G + t) * ncl + split) * (ATT_HD + 2);
            o[ATT_HD] = nst > 0 ? run_m[t] : -FLT_MAX;
            o[ATT_HD + 1] = run_l[t];
        }
        asm volatile("bar.sync 1, %0;" ::"n"(AS_CW * 32));
        if (t == 0) last_s = atomic_add_acq_rel_gpu(p.cnt + g * G, 1) == S - 1;  // releases the partial, acquires the others'
        asm volatile("bar.sync 1, %0;" ::"n"(AS_CW * 32));
        if (last_s) {
            // the fold, in split order: warp hh takes head hh, lane the dimensions lane + 32 k (k = 0..3: one 32-value
            // block each, quantized by the warp)
            if (wid < G) {
                const float* base = p.part + ((int64_t)g * G + wid) * ncl * (ATT_HD + 2);
                float M = -FLT_MAX, den = 0.f, num[4] = {0.f, 0.f, 0.f, 0.f};
                for (int c = 0; c < S; ++c) {
                    const float* src = base + (int64_t)c * (ATT_HD + 2);
                    const float mc = __ldcg(src + ATT_HD);
                    if (mc == -FLT_MAX) continue;  // an empty split
                    const float lc = __ldcg(src + ATT_HD + 1);
                    float vc[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) vc[k] = __ldcg(src + lane + 32 * k);
                    const float Mn = fmaxf(M, mc);
                    const float r = M == -FLT_MAX ? 0.f : expf(M - Mn), f = expf(mc - Mn);
                    den = den * r + f * lc;
#pragma unroll
                    for (int k = 0; k < 4; ++k) num[k] = fmaf(f, vc[k], num[k] * r);
                    M = Mn;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float o = num[k] / den;
                    const int64_t oi = ((int64_t)g * G + wid) * ATT_HD + lane + 32 * k;
                    p.out[oi] = o;
                    if (p.outq) {
                        float dsc;
                        if (p.outl) {
                            int8_t lv;
                            p.outq[oi] = quantize2_lane(o, dsc, lv);
                            p.outl[oi] = lv;
                        } else {
                            p.outq[oi] = quantize_lane(o, dsc);
                        }
                        if (lane == 0) p.outs[oi / 32] = dsc;
                    }
                }
            }
            if (t == 0) p.cnt[g * G] = 0;
        }
    }
}

// ==== arg-max and advance ========================================================================================

constexpr int AM_THREADS = 512;

__device__ __forceinline__ bool am_better(float v, int i, float bv, int bi) {
    return bi < 0 || v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(AM_THREADS) argmax_kernel(const float* __restrict__ x, int64_t n, float* bv_out,
                                                            int* bi_out, int* cnt, int32_t* tok, int32_t* pos,
                                                            const int* err, int ctx, L2Prefetch pf) {
    __shared__ float sv[AM_THREADS / 32];
    __shared__ int si[AM_THREADS / 32];
    __shared__ int last;
    issue_l2_prefetch(pf);
    griddep_wait();
    {  // row blockIdx.y of a batch: its logits, scratch, counter, token and position
        const int row = blockIdx.y;
        x += (int64_t)row * n;
        bv_out += (int64_t)row * gridDim.x;
        bi_out += (int64_t)row * gridDim.x;
        cnt += row;
        tok += row;
        if (pos) pos += row;
    }
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    float bv = -FLT_MAX;
    int bi = -1;
    for (int64_t i = (int64_t)blockIdx.x * AM_THREADS + t; i < n; i += (int64_t)gridDim.x * AM_THREADS) {
        const float v = x[i];
        if (am_better(v, (int)i, bv, bi)) {
            bv = v;
            bi = (int)i;
        }
    }
    auto reduce = [&](float& v, int& i) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, o);
            const int oi = __shfl_xor_sync(0xffffffffu, i, o);
            if (oi >= 0 && am_better(ov, oi, v, i)) {
                v = ov;
                i = oi;
            }
        }
    };
    reduce(bv, bi);
    if (lane == 0) {
        sv[wid] = bv;
        si[wid] = bi;
    }
    __syncthreads();
    if (wid == 0) {
        bv = lane < AM_THREADS / 32 ? sv[lane] : -FLT_MAX;
        bi = lane < AM_THREADS / 32 ? si[lane] : -1;
        reduce(bv, bi);
        if (lane == 0) {
            bv_out[blockIdx.x] = bv;
            bi_out[blockIdx.x] = bi;
            __threadfence();
            last = (atomicAdd(cnt, 1) == (int)gridDim.x - 1);
        }
    }
    __syncthreads();
    if (!last || wid != 0) return;
    __threadfence();
    bv = -FLT_MAX;
    bi = -1;
    for (int b = lane; b < (int)gridDim.x; b += 32) {
        const float v = __ldcg(bv_out + b);
        const int i = __ldcg(bi_out + b);
        if (i >= 0 && am_better(v, i, bv, bi)) {
            bv = v;
            bi = i;
        }
    }
    reduce(bv, bi);
    if (lane == 0) {
        const bool bad = (err && __ldcg(err) != 0) || (pos && (*pos < 0 || *pos >= ctx));
        if (!bad) {
            *tok = bi;
            if (pos) *pos = *pos + 1;
        }
        *cnt = 0;
    }
}

__global__ void rope_table_kernel(float* cos_t, float* sin_t, int ctx, int half, double theta) {
    const int64_t n = (int64_t)ctx * half;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t pos = i / half;
        const int j = (int)(i % half);
        const double ang = (double)pos * pow(theta, -2.0 * (double)j / (double)(2 * half));
        double s, c;
        sincos(ang, &s, &c);
        cos_t[i] = (float)c;
        sin_t[i] = (float)s;
    }
}

int attn_chunks(int ctx) {
    const int n = (ctx + ATT_CHUNK - 1) / ATT_CHUNK;
    return (n + ATT_CLUSTER - 1) / ATT_CLUSTER * ATT_CLUSTER;
}

int argmax_blocks(int64_t n) {
    int64_t b = (n + AM_THREADS * 4 - 1) / (AM_THREADS * 4);
    const int64_t cap = (int64_t)device_info().sms * 2;
    if (b > cap) b = cap;
    if (b < 1) b = 1;
    return (int)b;
}

// ==== a chunk of token rows ======================================================================================

// Row r of the residual stream is the embedding row of tokens[r] (an id outside [0, vocab) reads row 0 and sets
// error bit 1); posr[r] = *pos + r, the position row r takes (a row past the cache end sets bit 2, and its attention
// launch then writes and attends nothing).
__global__ void __launch_bounds__(256) chunk_setup_kernel(const int32_t* tokens, const float* embed, int64_t D,
                                                          int64_t vocab, const int32_t* pos, int ctx, int32_t* posr,
                                                          float* h, int* err) {
    const int r = blockIdx.x;
    const int32_t tk = tokens[r];
    const bool bad = tk < 0 || tk >= vocab;
    const float* src = embed + (bad ? 0 : (int64_t)tk) * D;
    float* dst = h + (int64_t)r * D;
    for (int64_t i = threadIdx.x; i < D; i += blockDim.x) dst[i] = __ldg(src + i);
    if (threadIdx.x == 0) {
        const int p = *pos + r;
        posr[r] = p;
        if (bad && err) atomicOr(err, 1);
        if ((p < 0 || p >= ctx) && err) atomicOr(err, 2);
    }
}

// The chunk's rows at their positions: per-head QK-norm and RoPE of every row's queries (into qr) and keys, and the
// keys and values appended to the caches, before any row attends.  A CTA per row, a warp per head vector, lane l
// holding dims l, l + 32, l + 64, l + 96 (so the rotation pairs (i, i + 64) sit in one lane).
__global__ void __launch_bounds__(256) chunk_append_kernel(const float* q, const float* k, const float* v,
                                                           const float* q_norm, const float* k_norm,
                                                           const float* cos_t, const float* sin_t, float eps,
                                                           const int32_t* posr, int heads, int kv, int ctx,
                                                           float* k_cache, float* v_cache, float* qr) {
    const int r = blockIdx.x, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int pos = posr[r];
    if (pos < 0 || pos >= ctx) return;  // flagged by the chunk setup
    for (int hv = wid; hv < heads + 2 * kv; hv += blockDim.x / 32) {
        if (hv >= heads + kv) {  // a value row: copied
            const int g = hv - heads - kv;
            const float* src = v + ((int64_t)r * kv + g) * ATT_HD;
            float* dst = v_cache + ((int64_t)g * ctx + pos) * ATT_HD;
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[lane + 32 * j] = src[lane + 32 * j];
            continue;
        }
        const bool isq = hv < heads;
        const float* src = isq ? q + ((int64_t)r * heads + hv) * ATT_HD : k + ((int64_t)r * kv + (hv - heads)) * ATT_HD;
        const float* w = isq ? q_norm : k_norm;
        float x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = src[lane + 32 * j];
        const float ss = group_sum<32>((x[0] * x[0] + x[2] * x[2]) + (x[1] * x[1] + x[3] * x[3]));
        const float inv = 1.0f / sqrtf(ss / (float)ATT_HD + eps);
        float y[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) y[j] = x[j] * inv * w[lane + 32 * j];
        // NeoX rotation of (i, i + 64): dims lane + 32j for j = 0, 1 pair with j = 2, 3
        float o[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = lane + 32 * j;
            const float cs = cos_t[(int64_t)pos * (ATT_HD / 2) + i], sn = sin_t[(int64_t)pos * (ATT_HD / 2) + i];
            o[j] = y[j] * cs - y[j + 2] * sn;
            o[j + 2] = y[j] * sn + y[j + 2] * cs;
        }
        float* dst = isq ? qr + ((int64_t)r * heads + hv) * ATT_HD
                         : k_cache + ((int64_t)(hv - heads) * ctx + pos) * ATT_HD;
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[lane + 32 * j] = o[j];
    }
}

// Causal attention of a chunk's rows, split over positions: CTA (key/value head g, position group pg, row block rb)
// takes rows rb*ACH_RB .. +ACH_RB-1 (every query head of the group: ACH_RB * G query vectors) against positions
// pg*ACH_GROUP*64 .. +ACH_GROUP*64-1 in chunks of 64, keeping a running (max, sum, weighted values) per query vector
// (online softmax, chunks in order); row r attends positions 0 .. posr[r].  The group's result (max, sum, 128
// weighted values) goes to part[r][head][pg] when the row had any position in the group.
// Scores: four lanes a position pair (a 32-dim quarter each, both key rows in registers, the next chunk's loaded once
// this chunk's scores are done), each query read from shared memory feeding both positions.
// Values: the chunk's value rows arrive in shared memory by cp.async while the scores are formed; thread (w, lane)
// owns dims 4*lane .. +3 of query vectors w, w + 8, ..., reading each value row once for all of them.
constexpr int ACH_RB = 8;      // rows per CTA
constexpr int ACH_GROUP = 2;   // 64-position chunks per CTA
constexpr int ACH_PAIRS = ACH_RB * ATT_MAXG;  // query vectors per CTA
constexpr int ACH_QS = 4 * ATT_QP;             // a query vector in shared memory: four padded 32-dim quarters
constexpr int ACH_PS = ATT_HD + 4;             // a group result: 128 weighted values, max, sum (16-byte rows)
constexpr int ACH_SS = 68;                     // a query vector's 64 scores (16-byte rows: four read at once)
constexpr size_t ACH_SMEM = (size_t)(64 * ATT_HD + ACH_PAIRS * ACH_QS + ACH_PAIRS * ACH_SS + 3 * ACH_PAIRS + 16) *
                            sizeof(float);

__global__ void __launch_bounds__(256, 2) chunk_attention_kernel(const float* qr, const float* k_cache,
                                                                 const float* v_cache, const int32_t* posr, int R,
                                                                 int heads, int kv, int ctx, float scale, float* part,
                                                                 int ngroups) {
    extern __shared__ __align__(16) float acs[];
    float* vs = acs;                           // [64][128]
    float* qs = vs + 64 * ATT_HD;              // [pairs][4][ATT_QP]
    float* sc = qs + ACH_PAIRS * ACH_QS;       // [pairs][ACH_SS]
    float* mrun = sc + ACH_PAIRS * ACH_SS;     // [pairs] running max
    float* lrun = mrun + ACH_PAIRS;            // [pairs] running sum
    float* fold = lrun + ACH_PAIRS;            // [pairs] rescale of this chunk
    int* lim = reinterpret_cast<int*>(fold + ACH_PAIRS);  // [ACH_RB] each row's last position
    const int g = blockIdx.x, pg = blockIdx.y, rb = blockIdx.z;
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int G = heads / kv;
    const int r0 = rb * ACH_RB, nr = min(ACH_RB, R - r0);
    if (nr <= 0) return;
    int maxpos = -1;
    for (int i = 0; i < nr; ++i) maxpos = max(maxpos, min(posr[r0 + i], ctx - 1));
    const int p_begin = pg * ACH_GROUP * 64;
    if (p_begin > maxpos) return;  // every row of the block ends before this group
    const int nchunk = min(ACH_GROUP, (maxpos - p_begin) / 64 + 1);
    // score role: warps w and w + 4 share positions 16*(w%4) .. +15 (two a lane group, dims 32*sub ..); warp w takes
    // query vectors 32*(w/4) .. +31
    const int sub = lane & 3, pa = 16 * (wid & 3) + 2 * (lane >> 2), pv0 = 32 * (wid >> 2);
    auto load_k = [&](int cc, float (&kr)[2][32]) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int p = p_begin + cc * 64 + pa + j;
            if (cc < nchunk && p <= maxpos) {
                const float* kp = k_cache + ((int64_t)g * ctx + p) * ATT_HD + sub * 32;
#pragma unroll
                for (int i = 0; i < 4; ++i) ld_f8_stream(kp + 8 * i, &kr[j][8 * i]);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) kr[j][i] = 0.f;
            }
        }
    };
    auto load_v = [&](int cc) {  // the chunk's value rows into vs by cp.async (rows past maxpos: zeros)
        for (int i = t; i < 64 * (ATT_HD / 4); i += blockDim.x) {
            const int row = i / (ATT_HD / 4), d4 = i % (ATT_HD / 4);
            const int p = p_begin + cc * 64 + row;
            float* dst = vs + row * ATT_HD + 4 * d4;
            if (p <= maxpos)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                             "l"(v_cache + ((int64_t)g * ctx + p) * ATT_HD + 4 * d4) : "memory");
            else
                *reinterpret_cast<float4*>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    float kr[2][32];
    load_k(0, kr);
    load_v(0);
    // the block's queries: pair = row_in_block * ATT_MAXG + head_in_group
    for (int i = t; i < ACH_PAIRS * ATT_HD; i += blockDim.x) {
        const int pr = i / ATT_HD, d = i % ATT_HD, rr = pr / ATT_MAXG, hh = pr % ATT_MAXG;
        const bool ok = rr < nr && hh < G;
        qs[pr * ACH_QS + (d >> 5) * ATT_QP + (d & 31)] =
            ok ? qr[((int64_t)(r0 + rr) * heads + g * G + hh) * ATT_HD + d] : 0.f;
    }
    for (int i = t; i < ACH_PAIRS; i += blockDim.x) {
        mrun[i] = -FLT_MAX;
        lrun[i] = 0.f;
    }
    if (t < ACH_RB) lim[t] = t < nr ? min(posr[r0 + t], ctx - 1) : -1;
    float4 acc[ACH_PAIRS / 8];
#pragma unroll
    for (int i = 0; i < ACH_PAIRS / 8; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    for (int cc = 0; cc < nchunk; ++cc) {
        const int p0 = p_begin + cc * 64;
        // scores of this warp's query vectors against the lane group's two positions (two vectors at a time)
        for (int pr0 = pv0; pr0 < pv0 + 32; pr0 += 2) {
            float a[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float4 q4 = reinterpret_cast<const float4*>(qs + (pr0 + u) * ACH_QS + sub * ATT_QP)[i];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        a[j][u] = fmaf(q4.x, kr[j][4 * i], a[j][u]);
                        a[j][u] = fmaf(q4.y, kr[j][4 * i + 1], a[j][u]);
                        a[j][u] = fmaf(q4.z, kr[j][4 * i + 2], a[j][u]);
                        a[j][u] = fmaf(q4.w, kr[j][4 * i + 3], a[j][u]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    a[j][u] += __shfl_xor_sync(0xffffffffu, a[j][u], 1);
                    a[j][u] += __shfl_xor_sync(0xffffffffu, a[j][u], 2);
                }
            if (sub == 0) {
                const int lm = lim[pr0 / ATT_MAXG];  // the two vectors share a row
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        sc[(pr0 + u) * ACH_SS + pa + j] = p0 + pa + j <= lm ? a[j][u] * scale : -FLT_MAX;
            }
        }
        __syncthreads();
        load_k(cc + 1, kr);  // the next chunk's keys, in flight during this chunk's softmax and values
        // softmax update per query vector (warp w takes vectors w, w + 8, ...)
        for (int pr = wid; pr < ACH_PAIRS; pr += 8) {
            const float s0 = sc[pr * ACH_SS + lane], s1 = sc[pr * ACH_SS + lane + 32];
            const float cm = warp_max(fmaxf(s0, s1));
            const float mo = mrun[pr];
            const float mn = fmaxf(mo, cm);
            float e0 = 0.f, e1 = 0.f, f = 1.f;
            if (mn != -FLT_MAX) {
                e0 = s0 == -FLT_MAX ? 0.f : expf(s0 - mn);
                e1 = s1 == -FLT_MAX ? 0.f : expf(s1 - mn);
                f = mo == -FLT_MAX ? 0.f : expf(mo - mn);
            }
            sc[pr * ACH_SS + lane] = e0;
            sc[pr * ACH_SS + lane + 32] = e1;
            const float cs = group_sum<32>(e0 + e1);
            if (lane == 0) {
                lrun[pr] = lrun[pr] * f + cs;
                mrun[pr] = mn;
                fold[pr] = f;
            }
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();  // weights, rescales and the chunk's value rows
#pragma unroll
        for (int i = 0; i < ACH_PAIRS / 8; ++i) {
            const float f = fold[wid + 8 * i];
            acc[i].x *= f;
            acc[i].y *= f;
            acc[i].z *= f;
            acc[i].w *= f;
        }
        for (int p = 0; p < 64; p += 4) {  // four value rows, and each vector's four weights in one read
            float4 v4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v4[j] = reinterpret_cast<const float4*>(vs + (p + j) * ATT_HD)[lane];
#pragma unroll
            for (int i = 0; i < ACH_PAIRS / 8; ++i) {
                const float4 e4 = *reinterpret_cast<const float4*>(sc + (wid + 8 * i) * ACH_SS + p);
                const float e[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i].x = fmaf(e[j], v4[j].x, acc[i].x);
                    acc[i].y = fmaf(e[j], v4[j].y, acc[i].y);
                    acc[i].z = fmaf(e[j], v4[j].z, acc[i].z);
                    acc[i].w = fmaf(e[j], v4[j].w, acc[i].w);
                }
            }
        }
        __syncthreads();  // the weights and value rows are read: the next chunk may overwrite them
        if (cc + 1 < nchunk) load_v(cc + 1);
    }
#pragma unroll
    for (int i = 0; i < ACH_PAIRS / 8; ++i) {
        const int pr = wid + 8 * i, rr = pr / ATT_MAXG, hh = pr % ATT_MAXG;
        if (rr >= nr || hh >= G) continue;
        float* dst = part + (((int64_t)(r0 + rr) * heads + g * G + hh) * ngroups + pg) * ACH_PS;
        reinterpret_cast<float4*>(dst)[lane] = acc[i];
        if (lane == 0) {
            dst[ATT_HD] = mrun[pr];
            dst[ATT_HD + 1] = lrun[pr];
        }
    }
}

// The same partials on the tensor cores.  CTA (key/value head g, position group pg, rows z*64 .. z*64+63) converts
// the group's 128 key and value rows once and then takes its row blocks of TCA_ROWS rows in turn: query vectors
// m = 8 * (row in block) + (head in group) (128 vectors: the MMA's M) against the group's positions, one pass each
// (no running rescale: the group is the unit the fold combines).  Every f32
// operand is split into two f16 parts, x = hi + lo (hi = x rounded to f16, lo = the remainder rounded to f16: the
// pair holds x to about 2^-22 relative), and the three products hi*hi + hi*lo + lo*hi are accumulated in f32 in
// tensor memory; the lo*lo term (about 2^-22 relative) is left out.
//  - S = Q K^T: 3 x 8 MMAs (M 128 query vectors, N 128 positions, K 16 dims each), the hi*hi products into TMEM
//    columns 0..127 and the cross products into 128..255, added in f32 when read (the tensor cores' accumulation
//    rounds each step; keeping the large terms apart from the small halves the steps that round them).
//  - Thread (vector m = 32 * (w % 4) + lane, positions 32 * (w / 4) ..) scales and masks its 32 scores (row r
//    attends positions 0 .. posr[r]), and with its vector's three other threads takes the max and the sum of the
//    weights e = exp(s - max); the weights go back, split the same way, as the A operand of the second product
//    (positions along K) over the queries' buffers.
//  - O = E V: 3 x 8 MMAs (N 128 dims, K 16 positions each), hi*hi into columns 256..383 and the cross products into
//    384..511; the value rows were transposed when converted (dims as B's rows, positions along K).
// Before the split each operand tile is scaled by a power of two (the weights by 2^14; queries, keys and values so
// that the tile's largest magnitude lies in [2^14, 2^15)), which keeps the lo parts normal f16 numbers; the results
// are scaled back exactly.  The partial (128 weighted values, max, sum) goes to part[r][head][pg] as
// chunk_attention_kernel writes it.  A tile holding an infinity or a NaN sets kErrHalfRange in the error word.
constexpr int TCA_ROWS = 16;                       // rows per row block
constexpr int TCA_BLOCKS = 4;                      // row blocks per CTA (keys and values converted once for them)
constexpr int TCA_M = TCA_ROWS * ATT_MAXG;         // query vectors per CTA: the MMA's M
constexpr int TCA_P = ACH_GROUP * 64;              // positions per CTA: the partials' position group
constexpr int TCA_THREADS = 512;
constexpr int TCA_TILE = 128 * ATT_HD * 2;         // bytes of an f16 operand tile of 128 rows x 128
constexpr uint32_t TCA_SBO = (ATT_HD / 8) * 128;   // bytes between its 8-row groups
constexpr size_t TCA_SMEM = 6 * (size_t)TCA_TILE + 2 * (size_t)TCA_M * 4 * sizeof(float);
constexpr int kErrHalfRange = 8;                   // error bit: a tensor-core attention tile that is not finite
static_assert(TCA_M == 128 && TCA_P == 128 && ATT_HD == 128, "one 128 x 128 tile each way");

__device__ __forceinline__ uint32_t tca_off(int r, int k8) {  // bytes of (row r, halves 8 * k8 .. 8 * k8 + 7)
    return (uint32_t)(r >> 3) * TCA_SBO + (uint32_t)k8 * 128 + (uint32_t)(r & 7) * 16;
}

__device__ __forceinline__ uint32_t half2_bits(__half a, __half b) {
    return (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
}

constexpr int TCA_PEXP = 14;  // the weights e (at most 1) are split as e * 2^14

// 2^e as a float, e in [-126, 127].
__device__ __forceinline__ float exp2_int(int e) { return __int_as_float((127 + e) << 23); }

// max(a, b), not a number when b is not one (so an operand's NaN reaches the tile maximum).
__device__ __forceinline__ float fmax_nan(float a, float b) { return b != b ? b : fmaxf(a, b); }

// Copies eight values to v and returns their largest magnitude.
__device__ __forceinline__ float load8_amax(const float (&x)[8], float (&v)[8]) {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = x[i];
        m = fmax_nan(m, fabsf(x[i]));
    }
    return m;
}

// The CTA's largest magnitude over the first n of every thread's xa (all threads call it; bits of non-negative
// floats order as unsigned integers, and a NaN's above every finite value's).
__device__ __forceinline__ float block_amax(const float (&xa)[4], int n, unsigned int* slot) {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (i < n) m = fmax_nan(m, xa[i]);
    unsigned int b = __float_as_uint(m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
    if ((threadIdx.x & 31) == 0) atomicMax(slot, b);
    __syncthreads();
    return __uint_as_float(*slot);
}

// The power of two that brings a tile's largest magnitude into [2^14, 2^15) (0 for an all-zero tile); a maximum that
// is not finite sets kErrHalfRange in the error word.
__device__ __forceinline__ int tile_exponent(float amax, int* err) {
    if (!(amax <= FLT_MAX)) {
        if (err && threadIdx.x == 0) atomicOr(err, kErrHalfRange);
        return 0;
    }
    if (amax == 0.f) return 0;
    const int e = 14 - ilogbf(amax);
    return e < -100 ? -100 : (e > 100 ? 100 : e);
}

// Eight f32 values times 2^e (exact) into f16 hi and lo parts: hi = the value rounded to f16, lo = the remainder
// rounded to f16 (one 16-byte core-matrix row each).
__device__ __forceinline__ void split8_scaled(const float (&x)[8], int e, uint4& hi, uint4& lo) {
    const float f = exp2_int(e);
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = x[2 * i] * f, b = x[2 * i + 1] * f;
        const __half h0 = __float2half_rn(a), h1 = __float2half_rn(b);
        const __half l0 = __float2half_rn(a - __half2float(h0)), l1 = __float2half_rn(b - __half2float(h1));
        h[i] = half2_bits(h0, h1);
        l[i] = half2_bits(l0, l1);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__global__ void __launch_bounds__(TCA_THREADS, 1) chunk_attention_tc_kernel(const float* qr, const float* k_cache,
                                                                            const float* v_cache,
                                                                            const int32_t* posr, int R, int heads,
                                                                            int kv, int ctx, float scale, float* part,
                                                                            int ngroups, int* err) {
    extern __shared__ __align__(1024) unsigned char tsm[];
    unsigned char* qh = tsm;                  // queries, then the weights E (hi parts)
    unsigned char* ql = tsm + TCA_TILE;       // (lo parts)
    unsigned char* kh = tsm + 2 * TCA_TILE;   // key rows
    unsigned char* kl = tsm + 3 * TCA_TILE;
    unsigned char* vh = tsm + 4 * TCA_TILE;   // value rows, transposed
    unsigned char* vl = tsm + 5 * TCA_TILE;
    float* pmax = reinterpret_cast<float*>(tsm + 6 * TCA_TILE);  // [vector][4] partial maxima
    float* psum = pmax + TCA_M * 4;                                // [vector][4] partial sums
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_base;
    __shared__ int lim[TCA_ROWS];
    __shared__ unsigned int amax[3];  // the query, key and value tiles' largest magnitudes (f32 bits)
    const int g = blockIdx.x, pg = blockIdx.y;
    const int t = threadIdx.x, w = t >> 5, lane = t & 31;
    const int G = heads / kv;
    const int rbeg = blockIdx.z * TCA_ROWS * TCA_BLOCKS, rend = min(R, rbeg + TCA_ROWS * TCA_BLOCKS);
    if (rend <= rbeg) return;
    int maxpos = -1;  // the last position any of the CTA's rows attends
    for (int i = rbeg; i < rend; ++i) maxpos = max(maxpos, min(posr[i], ctx - 1));
    const int p_begin = pg * TCA_P;
    if (p_begin > maxpos) return;  // every row ends before this group
    if (t == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    if (t < 3) amax[t] = 0u;
    if (w == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tc_smem(&tmem_base)),
                     "r"(512));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    __syncthreads();  // the tile maxima start at zero
    float xv[4][8];   // a thread's operand values between the tile's max and its split
    float xa[4];      // their largest magnitudes
    int evs = 0;
    // Each operand tile is scaled by a power of two before the split, so that its largest magnitude lies in
    // [2^14, 2^15): the lo parts of all but the tile's tiniest values stay normal f16 numbers.  The products are
    // scaled back exactly.
#pragma unroll
    for (int u = 0; u < TCA_P * 16 / TCA_THREADS; ++u) {  // key rows: position n, dims 8 * k8 ..
        const int task = t + u * TCA_THREADS, n = task >> 4, k8 = task & 15, p = p_begin + n;
        float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (p <= maxpos) {
            const float4* src = reinterpret_cast<const float4*>(k_cache + ((int64_t)g * ctx + p) * ATT_HD) + 2 * k8;
            const float4 a = __ldg(src), b = __ldg(src + 1);
            x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
        }
        xa[u] = load8_amax(x, xv[u]);
    }
    const int ek = tile_exponent(block_amax(xa, TCA_P * 16 / TCA_THREADS, &amax[1]), err);
#pragma unroll
    for (int u = 0; u < TCA_P * 16 / TCA_THREADS; ++u) {
        const int task = t + u * TCA_THREADS, n = task >> 4, k8 = task & 15;
        uint4 hi, lo;
        split8_scaled(xv[u], ek, hi, lo);
        *reinterpret_cast<uint4*>(kh + tca_off(n, k8)) = hi;
        *reinterpret_cast<uint4*>(kl + tca_off(n, k8)) = lo;
    }
    static_assert((ATT_HD / 4) * (TCA_P / 8) == TCA_THREADS, "one value task a thread");
    {  // values: dims 4 * d4 .. +3, positions 8 * p8 .. +7 (transposed: dims as B's rows)
        const int d4 = t & (ATT_HD / 4 - 1), p8 = t / (ATT_HD / 4);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int p = p_begin + 8 * p8 + i;
            const float4 v4 = p <= maxpos ? __ldg(reinterpret_cast<const float4*>(v_cache + ((int64_t)g * ctx + p) * ATT_HD) + d4)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
            xv[0][i] = v4.x, xv[1][i] = v4.y, xv[2][i] = v4.z, xv[3][i] = v4.w;
        }
        float mv = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i) mv = fmax_nan(mv, fabsf(xv[j][i]));
        xa[0] = mv;
        const int ev = tile_exponent(block_amax(xa, 1, &amax[2]), err);
        evs = ev;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 hi, lo;
            split8_scaled(xv[j], ev, hi, lo);
            *reinterpret_cast<uint4*>(vh + tca_off(4 * d4 + j, p8)) = hi;
            *reinterpret_cast<uint4*>(vl + tca_off(4 * d4 + j, p8)) = lo;
        }
    }
    const uint32_t tmem = tmem_base;
    const uint32_t idesc = tc_idesc_f16(128, 128);
    bool ok = true;
    for (int r0 = rbeg; r0 < rend; r0 += TCA_ROWS) {  // the row blocks: the keys and values stay converted
        const int nr = min(TCA_ROWS, rend - r0);
        int bmax = -1;
        for (int i = 0; i < nr; ++i) bmax = max(bmax, min(posr[r0 + i], ctx - 1));
        if (p_begin > bmax) continue;  // every row of the block ends before this group (CTA-uniform)
        if (t < TCA_ROWS) lim[t] = t < nr ? min(posr[r0 + t], ctx - 1) : -1;
        if (t == 0) amax[0] = 0u;
        __syncthreads();  // the block's limits and its tile maximum; the previous block's products are read
#pragma unroll
        for (int u = 0; u < TCA_M * 16 / TCA_THREADS; ++u) {  // queries: vector m, dims 8 * k8 ..
            const int task = t + u * TCA_THREADS, m = task >> 4, k8 = task & 15, rr = m >> 3, hh = m & 7;
            float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (rr < nr && hh < G) {
                const float4* src = reinterpret_cast<const float4*>(qr + ((int64_t)(r0 + rr) * heads + g * G + hh) * ATT_HD) + 2 * k8;
                const float4 a = src[0], b = src[1];
                x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
            }
            xa[u] = load8_amax(x, xv[u]);
        }
        const int eq = tile_exponent(block_amax(xa, TCA_M * 16 / TCA_THREADS, &amax[0]), err);
#pragma unroll
        for (int u = 0; u < TCA_M * 16 / TCA_THREADS; ++u) {
            const int task = t + u * TCA_THREADS, m = task >> 4, k8 = task & 15;
            uint4 hi, lo;
            split8_scaled(xv[u], eq, hi, lo);
            *reinterpret_cast<uint4*>(qh + tca_off(m, k8)) = hi;
            *reinterpret_cast<uint4*>(ql + tca_off(m, k8)) = lo;
        }
        const float s_back = exp2_int(-eq) * exp2_int(-ek) * scale;  // scores: D * 2^-(eq + ek), then the 1/sqrt(hd) scale
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the operands, to the tensor cores
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (t == 0 && ok) {
#pragma unroll 1
            for (int j = 0; j < ATT_HD / 16; ++j) {  // K = 16 dims: two core matrices along K
                const int o = j * 256;
                tc_mma_f16(tmem, tc_desc(qh + o, TCA_SBO), tc_desc(kh + o, TCA_SBO), idesc, j > 0 ? 1u : 0u);
                tc_mma_f16(tmem + 128, tc_desc(qh + o, TCA_SBO), tc_desc(kl + o, TCA_SBO), idesc, j > 0 ? 1u : 0u);
                tc_mma_f16(tmem + 128, tc_desc(ql + o, TCA_SBO), tc_desc(kh + o, TCA_SBO), idesc, 1u);
            }
            tc_commit(&bar);
        }
        if (ok) ok = __syncthreads_and(mbar_wait(&bar, 0, err) ? 1 : 0) != 0;  // (each block completes two phases)
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const int lq = w & 3, cq = w >> 2, m = 32 * lq + lane, rr = m >> 3, hh = m & 7;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * lq) << 16);
        const int lm = lim[rr];
        float s[32];
        {
            uint32_t sv[32], sx[32];
            tc_ld32(lane_base + 32 * cq, sv);        // hi * hi
            tc_ld32(lane_base + 128 + 32 * cq, sx);  // hi * lo + lo * hi
            tc_wait_ld();
            float mx = -FLT_MAX;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float d = __uint_as_float(sv[i]) + __uint_as_float(sx[i]);
                s[i] = p_begin + 32 * cq + i <= lm ? d * s_back : -FLT_MAX;
                mx = fmaxf(mx, s[i]);
            }
            pmax[m * 4 + cq] = mx;
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();  // every partial max; the first product is read (its operands may be overwritten)
        const float M = fmaxf(fmaxf(pmax[m * 4], pmax[m * 4 + 1]), fmaxf(pmax[m * 4 + 2], pmax[m * 4 + 3]));
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            s[i] = (M == -FLT_MAX || s[i] == -FLT_MAX) ? 0.f : expf(s[i] - M);
            sum += s[i];
        }
        psum[m * 4 + cq] = sum;
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8) {  // the weights (at most 1) times 2^14, positions 32 * cq + 8 * k8 .., as A
            uint4 hi, lo;
            float x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = s[8 * k8 + i];
            split8_scaled(x, TCA_PEXP, hi, lo);
            *reinterpret_cast<uint4*>(qh + tca_off(m, 4 * cq + k8)) = hi;
            *reinterpret_cast<uint4*>(ql + tca_off(m, 4 * cq + k8)) = lo;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (t == 0 && ok) {
#pragma unroll 1
            for (int j = 0; j < TCA_P / 16; ++j) {  // K = 16 positions
                const int o = j * 256;
                tc_mma_f16(tmem + 256, tc_desc(qh + o, TCA_SBO), tc_desc(vh + o, TCA_SBO), idesc, j > 0 ? 1u : 0u);
                tc_mma_f16(tmem + 384, tc_desc(qh + o, TCA_SBO), tc_desc(vl + o, TCA_SBO), idesc, j > 0 ? 1u : 0u);
                tc_mma_f16(tmem + 384, tc_desc(ql + o, TCA_SBO), tc_desc(vh + o, TCA_SBO), idesc, 1u);
            }
            tc_commit(&bar);
        }
        if (ok) ok = __syncthreads_and(mbar_wait(&bar, 1, err) ? 1 : 0) != 0;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (ok) {
            uint32_t ov[32], ox[32];
            tc_ld32(lane_base + 256 + 32 * cq, ov);  // hi * hi
            tc_ld32(lane_base + 384 + 32 * cq, ox);  // hi * lo + lo * hi
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) + __uint_as_float(ox[i]));
            if (rr < nr && hh < G) {
                float* dst = part + (((int64_t)(r0 + rr) * heads + g * G + hh) * ngroups + pg) * ACH_PS;
                const float o_back = exp2_int(-TCA_PEXP) * exp2_int(-evs);  // exact
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    reinterpret_cast<float4*>(dst + 32 * cq)[i] =
                        make_float4(__uint_as_float(ov[4 * i]) * o_back, __uint_as_float(ov[4 * i + 1]) * o_back,
                                    __uint_as_float(ov[4 * i + 2]) * o_back, __uint_as_float(ov[4 * i + 3]) * o_back);
                if (cq == 0) {
                    dst[ATT_HD] = M;
                    dst[ATT_HD + 1] = ((psum[m * 4] + psum[m * 4 + 1]) + psum[m * 4 + 2]) + psum[m * 4 + 3];
                }
            }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();  // every thread has read the block's results: the next block may overwrite them
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (w == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
}

// Row r, head h: the position groups' results folded in group order, out = num / den, and its int8 form.  A warp
// per (row, head), lane l the dims l, l + 32, l + 64, l + 96.  The groups' maxima and sums are read a group a lane
// (32 at a time) and passed along by shuffles; each group's values are then added in group order, four groups'
// loads in flight at once.
__global__ void __launch_bounds__(256) chunk_attn_fold_kernel(const float* part, const int32_t* posr, int R, int heads,
                                                              int ctx, int ngroups, float* out, int8_t* outq,
                                                              int8_t* outl, float* outs) {
    const int wg = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (wg >= R * heads) return;
    const int r = wg / heads;
    const int pos = posr[r];
    if (pos < 0 || pos >= ctx) return;
    const int ng = min(ngroups, pos / (ACH_GROUP * 64) + 1);
    const float* base = part + (int64_t)wg * ngroups * ACH_PS;
    float M = -FLT_MAX;
    for (int c = lane; c < ng; c += 32) M = fmaxf(M, __ldcg(base + (int64_t)c * ACH_PS + ATT_HD));
    M = warp_max(M);
    float num[4] = {0.f, 0.f, 0.f, 0.f}, den = 0.f;
    for (int c0 = 0; c0 < ng; c0 += 32) {
        const int nb = min(32, ng - c0);
        float f = 0.f, l = 0.f;
        int live = 0;
        if (lane < nb) {
            const float* b = base + (int64_t)(c0 + lane) * ACH_PS;
            const float mc = __ldcg(b + ATT_HD);
            if (mc != -FLT_MAX) {
                live = 1;
                f = expf(mc - M);
                l = __ldcg(b + ATT_HD + 1);
            }
        }
        for (int cc = 0; cc < nb; cc += 4) {
            float v[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float* b = base + (int64_t)(c0 + cc + u) * ACH_PS;
#pragma unroll
                for (int j = 0; j < 4; ++j) v[u][j] = cc + u < nb ? __ldcg(b + lane + 32 * j) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int src = (cc + u) & 31;
                const float fu = __shfl_sync(0xffffffffu, f, src), lu = __shfl_sync(0xffffffffu, l, src);
                const int lv = __shfl_sync(0xffffffffu, live, src);
                if (cc + u < nb && lv) {  // warp-uniform
                    den = fmaf(fu, lu, den);
#pragma unroll
                    for (int j = 0; j < 4; ++j) num[j] = fmaf(fu, v[u][j], num[j]);
                }
            }
        }
    }
    // the partials' values sit in float4 order (lane l held dims 4l..4l+3): dim d is at index d
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float o = num[j] / den;
        const int64_t oi = (int64_t)wg * ATT_HD + lane + 32 * j;
        out[oi] = o;
        if (outq) {
            float dsc;
            if (outl) {
                int8_t lv;
                outq[oi] = quantize2_lane(o, dsc, lv);
                outl[oi] = lv;
            } else {
                outq[oi] = quantize_lane(o, dsc);
            }
            if (lane == 0) outs[oi / 32] = dsc;
        }
    }
}

// *pos += add, unless the step's error word is set.
__global__ void pos_add_kernel(int32_t* pos, int add, const int* err) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && !(err && *err)) *pos += add;
}

}  // namespace

int kStreamedBatchAttention = 8;

void attention_scratch(const AttnCall& c, size_t* bytes, size_t* counters) {
    const int G = c.heads / c.kv;
    const int B = c.batch > 1 ? c.batch : 1;
    *bytes = (size_t)B * c.kv * G * (attn_chunks(c.ctx) / ATT_CLUSTER) * (ATT_HD + 2) * sizeof(float);
    *counters = (size_t)B * c.kv * G;
}

cudaError_t launch_attention(const AttnCall& c, Carve& ws, cudaStream_t st) {
    AttnParams p = {};
    p.q = c.q;
    p.k = c.k;
    p.v = c.v;
    p.q_norm = c.q_norm;
    p.k_norm = c.k_norm;
    p.cos_t = c.cos_t;
    p.sin_t = c.sin_t;
    p.eps = c.eps;
    p.err = c.err;
    p.k_cache = c.k_cache;
    p.v_cache = c.v_cache;
    p.pos = c.pos;
    p.heads = c.heads;
    p.kv = c.kv;
    p.ctx = c.ctx;
    p.G = c.heads / c.kv;
    p.scale = (float)(1.0 / sqrt((double)c.hd));
    p.out = c.out;
    p.outq = c.outq;
    p.outl = c.outl;
    p.outs = c.outs;
    p.nch_max = attn_chunks(c.ctx);
    p.ncl_max = p.nch_max / ATT_CLUSTER;
    p.cache_stride = c.cache_stride;
    p.pf = c.pf;
    size_t bytes = 0, cnt = 0;
    attention_scratch(c, &bytes, &cnt);
    p.part = ws.take<float>(bytes / sizeof(float));
    p.cnt = ws.take_counters(cnt);
    if (ws.overflow) return cudaErrorMemoryAllocation;
    const int B = c.batch > 1 ? c.batch : 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c.kv, p.nch_max, B);
    cfg.blockDim = dim3(ATT_THREADS);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = ATT_CLUSTER;
    attr[0].val.clusterDim.z = 1;
    int na = 1;
    if (c.pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (B > 1 && kStreamedBatchAttention && B >= kStreamedBatchAttention) {
        // the streamed form: as many splits of the positions as the chunked form has clusters of 8 chunks (one scratch
        // slot each), no clusters
        static const cudaError_t set = cudaFuncSetAttribute(attention_stream_kernel,
                                                            cudaFuncAttributeMaxDynamicSharedMemorySize, (int)AS_SMEM);
        if (set != cudaSuccess) return set;
        cfg.gridDim = dim3(p.ncl_max, c.kv, B);
        cfg.blockDim = dim3(AS_THREADS);
        cfg.dynamicSmemBytes = AS_SMEM;
        cfg.attrs = attr + 1;
        cfg.numAttrs = na - 1;
        return cudaLaunchKernelEx(&cfg, attention_stream_kernel, p);
    }
    return B > 1 ? cudaLaunchKernelEx(&cfg, attention_kernel<true>, p) : cudaLaunchKernelEx(&cfg, attention_kernel<false>, p);
}

void argmax_scratch(const ArgmaxCall& c, size_t* bytes, size_t* counters) {
    const int rows = c.rows > 1 ? c.rows : 1;
    *bytes = (size_t)argmax_blocks(c.n) * 8 * rows + 256;
    *counters = rows;
}

cudaError_t launch_argmax(const ArgmaxCall& c, Carve& ws, cudaStream_t st) {
    const int blocks = argmax_blocks(c.n);
    const int rows = c.rows > 1 ? c.rows : 1;
    if (rows > 65535) return cudaErrorInvalidValue;
    float* bv = ws.take<float>((size_t)blocks * rows);
    int* bi = ws.take<int>((size_t)blocks * rows);
    int* cnt = ws.take_counters(rows);
    if (ws.overflow) return cudaErrorMemoryAllocation;
    return launch(argmax_kernel, dim3(blocks, rows), dim3(AM_THREADS), 0, st, c.pdl, c.x, c.n, bv, bi, cnt, c.tok,
                  c.pos, c.err, c.ctx, c.pf);
}

cudaError_t launch_rope_table(float* cos_t, float* sin_t, int ctx, int half, double theta, cudaStream_t st) {
    rope_table_kernel<<<256, 256, 0, st>>>(cos_t, sin_t, ctx, half, theta);
    return cudaGetLastError();
}

cudaError_t launch_chunk_setup(const int32_t* tokens, int64_t rows, const float* embed, int64_t D, int64_t vocab,
                               const int32_t* pos, int ctx, int32_t* posr, float* h, int* err, cudaStream_t st) {
    if (rows < 1) return cudaSuccess;
    chunk_setup_kernel<<<(unsigned)rows, 256, 0, st>>>(tokens, embed, D, vocab, pos, ctx, posr, h, err);
    return cudaGetLastError();
}

cudaError_t launch_pos_add(int32_t* pos, int add, const int* err, cudaStream_t st) {
    pos_add_kernel<<<1, 32, 0, st>>>(pos, add, err);
    return cudaGetLastError();
}

// Whether a prefill chunk's attention runs on the tensor cores (q8_set_tensor_core_attention).
int kChunkAttnTensorCores = 1;

int chunk_attn_groups(int ctx) { return (ctx + ACH_GROUP * 64 - 1) / (ACH_GROUP * 64); }

void chunk_attention_scratch(int64_t rows, int heads, int ctx, size_t* bytes) {
    *bytes = (size_t)rows * heads * chunk_attn_groups(ctx) * ACH_PS * sizeof(float) +
             (size_t)rows * heads * ATT_HD * sizeof(float);
}

cudaError_t launch_chunk_attention(const ChunkAttnCall& c, Carve& ws, cudaStream_t st) {
    if (c.hd != ATT_HD || c.heads % c.kv || c.heads / c.kv > ATT_MAXG || c.rows < 1) return cudaErrorInvalidValue;
    const int ng = chunk_attn_groups(c.ctx);
    float* qr = ws.take<float>((size_t)c.rows * c.heads * ATT_HD);
    float* part = ws.take<float>((size_t)c.rows * c.heads * ng * ACH_PS);
    if (ws.overflow) return cudaErrorMemoryAllocation;
    chunk_append_kernel<<<(unsigned)c.rows, 256, 0, st>>>(c.q, c.k, c.v, c.q_norm, c.k_norm, c.cos_t, c.sin_t, c.eps,
                                                          c.posr, c.heads, c.kv, c.ctx, c.k_cache, c.v_cache, qr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const float scale = (float)(1.0 / sqrt((double)c.hd));
    if (kChunkAttnTensorCores) {
        e = cudaFuncSetAttribute(chunk_attention_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TCA_SMEM);
        if (e != cudaSuccess) return e;
        const int rows_per_cta = TCA_ROWS * TCA_BLOCKS;
        const dim3 grid((unsigned)c.kv, (unsigned)ng, (unsigned)((c.rows + rows_per_cta - 1) / rows_per_cta));
        chunk_attention_tc_kernel<<<grid, TCA_THREADS, TCA_SMEM, st>>>(qr, c.k_cache, c.v_cache, c.posr, (int)c.rows,
                                                                       c.heads, c.kv, c.ctx, scale, part, ng, c.err);
    } else {
        e = cudaFuncSetAttribute(chunk_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ACH_SMEM);
        if (e != cudaSuccess) return e;
        const dim3 grid((unsigned)c.kv, (unsigned)ng, (unsigned)((c.rows + ACH_RB - 1) / ACH_RB));
        chunk_attention_kernel<<<grid, 256, ACH_SMEM, st>>>(qr, c.k_cache, c.v_cache, c.posr, (int)c.rows, c.heads,
                                                           c.kv, c.ctx, scale, part, ng);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t warps = c.rows * c.heads;
    chunk_attn_fold_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(part, c.posr, (int)c.rows, c.heads, c.ctx, ng,
                                                                       c.out, c.outq, c.outl, c.outs);
    return cudaGetLastError();
}

}  // namespace q8

