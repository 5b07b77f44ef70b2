/*
 * synth.c -- host implementation of the counter-based input generator.
 * Definitions are stated in synth.h.  Portable C99: no intrinsics, no
 * reliance on char signedness, identical results on x86_64 and aarch64 for
 * the integer streams and the fp16 scales (IEEE double, round-to-nearest).
 * The Box-Muller normals call libm log/cos; they are generated on the host
 * only and copied to the device, so both sides always see the same bytes.
 */
#include "synth.h"

#include <math.h>
#include <string.h>

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ull

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64((seed << 32) | (stream & 0xFFFFFFFFull));
}

uint64_t synth_draw(uint64_t seed, uint64_t stream, uint64_t i) {
  return mix64(stream_key(seed, stream) + (i + 1) * SYNTH_GOLDEN);
}

void synth_int8(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n, int8_t *out) {
  uint64_t key = stream_key(seed, stream);
  for (uint64_t j = 0; j < n; ++j) {
    uint64_t r = mix64(key + (first + j + 1) * SYNTH_GOLDEN);
    int v = -127 + (int)(((r >> 40) * 255u) >> 24);
    out[j] = (int8_t)v;
  }
}

void synth_code2(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n, uint8_t *out) {
  uint64_t key = stream_key(seed, stream);
  for (uint64_t j = 0; j < n; ++j) {
    uint64_t r = mix64(key + (first + j + 1) * SYNTH_GOLDEN);
    out[j] = (uint8_t)(r >> 56);
  }
}

uint16_t synth_f64_to_f16(double v) {
  uint16_t sign = signbit(v) ? 0x8000u : 0u;
  double a = fabs(v);
  if (isnan(v)) return 0x7E00u;
  /* 65520 is the midpoint between the largest finite fp16 (65504) and 2^16. */
  if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e); /* a = m * 2^e, m in [0.5, 1): the leading bit is 2^(e-1) */
  int lead = e - 1;
  if (lead < -14) {
    /* subnormal range: units of 2^-24 */
    double q = rint(ldexp(a, 24)); /* exact scaling, then ties-to-even */
    return (uint16_t)(sign | (uint16_t)q); /* q == 1024 gives the smallest normal */
  }
  double m = rint(ldexp(a, 10 - lead)); /* in [1024, 2048] */
  if (m >= 2048.0) {
    m = 1024.0;
    lead += 1;
  }
  if (lead > 15) return (uint16_t)(sign | 0x7C00u);
  uint16_t bits = (uint16_t)(((lead + 15) << 10) | ((uint16_t)m - 1024u));
  return (uint16_t)(sign | bits);
}

void synth_scale_f16(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n,
                     double denom, uint16_t *out) {
  uint64_t key = stream_key(seed, stream);
  for (uint64_t j = 0; j < n; ++j) {
    uint64_t r = mix64(key + (first + j + 1) * SYNTH_GOLDEN);
    double u = (double)(r >> 11) * 0x1.0p-53;
    out[j] = synth_f64_to_f16((0.5 + u) / denom);
  }
}

void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n,
                      double mean, double stddev, float *out) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t key = stream_key(seed, stream);
  for (uint64_t j = 0; j < n; ++j) {
    uint64_t i = first + j;
    uint64_t r1 = mix64(key + (2 * i + 1) * SYNTH_GOLDEN);
    uint64_t r2 = mix64(key + (2 * i + 2) * SYNTH_GOLDEN);
    double u1 = ((double)(r1 >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
    double u2 = (double)(r2 >> 11) * 0x1.0p-53;         /* [0, 1) */
    double z = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
    out[j] = (float)(mean + stddev * z);
  }
}

void synth_zipf_offset(uint64_t seed, uint64_t stream, uint32_t n_expert, double beta,
                       double a, float *out) {
  /* rank[e] in 1..E, a Fisher-Yates shuffle driven by the counter stream */
  uint32_t rank_buf[4096];
  uint32_t E = n_expert > 4096 ? 4096 : n_expert;
  for (uint32_t e = 0; e < E; ++e) rank_buf[e] = e + 1;
  for (uint32_t i = E; i > 1; --i) {
    uint64_t r = synth_draw(seed, stream, i);
    uint32_t j = (uint32_t)(r % i);
    uint32_t t = rank_buf[i - 1];
    rank_buf[i - 1] = rank_buf[j];
    rank_buf[j] = t;
  }
  for (uint32_t e = 0; e < E; ++e) out[e] = (float)(-beta * a * log((double)rank_buf[e]));
}
