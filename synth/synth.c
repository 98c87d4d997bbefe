/*
 * Seeded synthetic inputs: a counter-based generator shared by the tests and the benchmark.
 *
 * This file holds no arithmetic of the method: it only draws numbers.  Both the CPU oracle's callers and the CUDA
 * path's callers take their inputs from here, so the two sides always see identical bytes.
 *
 * Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014).
 * Its output function ("mix64", the variant-13 finaliser) is applied to a Weyl sequence; here the sequence is indexed
 * directly, so element i of a tensor is an independent function of (seed, tensor id, i):
 *
 *     key(seed, tensor) = mix64(mix64(seed + GAMMA) + (tensor + 1) * GAMMA)
 *     u64(seed, tensor, i) = mix64(key + (i + 1) * GAMMA)            GAMMA = 0x9E3779B97F4A7C15
 *
 * Derived draws:
 *     int8 weight      q = (u mod 255) - 127                     in [-127, 127]
 *     uniform [0,1)    (u >> 11) * 2^-53
 *     normal N(0,1)    Box-Muller (G. Box, M. Muller 1958) on two uniforms of draws 2i and 2i+1, cosine branch, f64
 *     f32 value        (float)(add + mul * z)  or  (float)(add + mul * |z|)
 *
 * Large fills are split over POSIX threads; the result does not depend on the thread count.
 */
#include "synth.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t tensor) { return mix64(mix64(seed + GAMMA) + (tensor + 1) * GAMMA); }

uint64_t synth_u64(uint64_t seed, uint64_t tensor, uint64_t i) { return mix64(synth_key(seed, tensor) + (i + 1) * GAMMA); }

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GAMMA); }

static inline double uniform53(uint64_t u) { return (double)(u >> 11) * 0x1.0p-53; }

static inline double normal_at(uint64_t key, uint64_t i) {
    /* u1 in (0, 1] keeps the logarithm finite; u2 in [0, 1). */
    double u1 = ((double)(draw(key, 2 * i) >> 11) + 1.0) * 0x1.0p-53;
    double u2 = uniform53(draw(key, 2 * i + 1));
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

double synth_normal(uint64_t seed, uint64_t tensor, uint64_t i) { return normal_at(synth_key(seed, tensor), i); }

/* ---- threaded fills -------------------------------------------------------------------------------------------- */

typedef struct {
    int kind; /* 0: int8, 1: normal f32 */
    uint64_t key, start, end, offset;
    double mul, add;
    int absval;
    void *out;
} job_t;

static void run_job(const job_t *j) {
    if (j->kind == 0) {
        int8_t *o = (int8_t *)j->out;
        for (uint64_t i = j->start; i < j->end; ++i) o[i] = (int8_t)((int)(draw(j->key, i + j->offset) % 255u) - 127);
    } else {
        float *o = (float *)j->out;
        for (uint64_t i = j->start; i < j->end; ++i) {
            double z = normal_at(j->key, i + j->offset);
            if (j->absval) z = fabs(z);
            o[i] = (float)(j->add + j->mul * z);
        }
    }
}

static void *thread_main(void *p) {
    run_job((const job_t *)p);
    return NULL;
}

static void fill(job_t base, uint64_t n, int threads) {
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if (n < (1u << 16) || threads == 1) {
        base.start = 0;
        base.end = n;
        run_job(&base);
        return;
    }
    pthread_t tid[256];
    int live[256];
    job_t jobs[256];
    for (int t = 0; t < threads; ++t) {
        jobs[t] = base;
        jobs[t].start = n * (uint64_t)t / (uint64_t)threads;
        jobs[t].end = n * (uint64_t)(t + 1) / (uint64_t)threads;
        live[t] = pthread_create(&tid[t], NULL, thread_main, &jobs[t]) == 0;
        if (!live[t]) run_job(&jobs[t]); /* no thread available: do this share here */
    }
    for (int t = 0; t < threads; ++t)
        if (live[t]) pthread_join(tid[t], NULL);
}

void synth_fill_i8(uint64_t seed, uint64_t tensor, uint64_t offset, uint64_t n, int8_t *out, int threads) {
    job_t j = {0};
    j.kind = 0;
    j.key = synth_key(seed, tensor);
    j.offset = offset;
    j.out = out;
    fill(j, n, threads);
}

void synth_fill_f32(uint64_t seed, uint64_t tensor, uint64_t offset, uint64_t n, double mul, double add, int absval,
                    float *out, int threads) {
    job_t j = {0};
    j.kind = 1;
    j.key = synth_key(seed, tensor);
    j.offset = offset;
    j.mul = mul;
    j.add = add;
    j.absval = absval;
    j.out = out;
    fill(j, n, threads);
}
