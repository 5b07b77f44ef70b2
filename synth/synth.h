/*
 * synth.h -- seeded, counter-based synthetic inputs for the routed-MoE layer.
 *
 * This module only draws numbers.  It holds none of the layer's arithmetic
 * (no scoring, selection, quantisation or dot products), so the CPU oracle and
 * the CUDA library can both be fed from it without sharing any of the method.
 *
 * Generator: every value is a pure function of (seed, stream, index).
 *   key     = mix64((seed << 32) | stream)            (seed, stream < 2^32)
 *   draw(i) = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)
 * where mix64 is the public-domain SplitMix64 finaliser (S. Vigna).
 * Derived values:
 *   int8   : -127 + ((draw >> 40) * 255 >> 24)           in [-127, 127]
 *   code2  : draw >> 56  (one byte = four 2-bit codes, uniform)
 *   unit53 : (draw >> 11) * 2^-53                          in [0, 1)
 *   scale  : fp16_rn((0.5 + unit53) / denom)               denom given by caller
 *   normal : Box-Muller, cosine branch, draws 2i and 2i+1 (host only)
 * The device fill kernels in synth_dev.cu implement the same definitions.
 */
#ifndef SYNTH_H
#define SYNTH_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

uint64_t synth_draw(uint64_t seed, uint64_t stream, uint64_t i);
void synth_int8(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n, int8_t *out);
void synth_code2(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n, uint8_t *out);
void synth_scale_f16(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n,
                     double denom, uint16_t *out);
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n,
                      double mean, double stddev, float *out);
/* Zipf-style popularity offset: a seeded permutation assigns each expert a
 * rank r in 1..E, and the offset is -beta * a * ln(r). */
void synth_zipf_offset(uint64_t seed, uint64_t stream, uint32_t n_expert, double beta,
                       double a, float *out);
/* Round a double to the nearest fp16 (ties to even); returns the bit pattern. */
uint16_t synth_f64_to_f16(double v);

#ifdef __cplusplus
}
#endif
#endif
