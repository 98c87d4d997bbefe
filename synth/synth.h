/* Seeded synthetic inputs (counter-based SplitMix64); see synth.c for the definition of every draw. */
#ifndef SYNTH_H
#define SYNTH_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

uint64_t synth_key(uint64_t seed, uint64_t tensor);
/* Draw i of tensor `tensor` under `seed`. */
uint64_t synth_u64(uint64_t seed, uint64_t tensor, uint64_t i);
/* The i-th N(0,1) value of a tensor (Box-Muller over draws 2i and 2i+1). */
double synth_normal(uint64_t seed, uint64_t tensor, uint64_t i);
/* out[j] = (u(offset + j) mod 255) - 127 for j < n. */
void synth_fill_i8(uint64_t seed, uint64_t tensor, uint64_t offset, uint64_t n, int8_t *out, int threads);
/* out[j] = (float)(add + mul * z) (or |z| when absval) with z the (offset + j)-th normal, for j < n. */
void synth_fill_f32(uint64_t seed, uint64_t tensor, uint64_t offset, uint64_t n, double mul, double add, int absval,
                    float *out, int threads);

#ifdef __cplusplus
}
#endif
#endif
