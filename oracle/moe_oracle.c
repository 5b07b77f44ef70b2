/*
 * moe_oracle.c -- the CPU oracle of the routed-MoE layer (test infrastructure).
 *
 * Straight loops, no blocking or fusion: a full scan per top-k slot, a
 * counting sort for the permutation, scalar int32 block dots and fp64 sums
 * in block order.  Floating point that decides an integer (the routing score,
 * the int8 codes of x and of h) is computed in fp32, the precision the CUDA
 * library uses for those decisions; every other quantity is fp64.
 * Build: cc -std=c99 -O2 -ffp-contract=off -fPIC -shared (no fused
 * multiply-adds other than the explicit fmaf calls in ora_spec_exp).
 * Definitions and page citations: oracle.h.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ spec-exp
 * e(x) for the router's sigmoid, defined so that any IEEE-754 fp32 machine
 * gets the same bits: clamp x to [-86, 88]; n = rint(x * log2(e)); Cody-Waite
 * reduction r = (x - n*C1) - n*C2 with C1 = 355/512 (exact products) and
 * C2 = fp32(ln2 - C1) (the split of Cody & Waite as used in Cephes);
 * p = degree-7 Taylor polynomial of e^r, coefficients fp32(1/k!), Horner with
 * fmaf; result p * 2^n with 2^n built exactly (n stays in [-124, 127]). */
float ora_spec_exp(float x) {
  const float log2e = 0x1.715476p+0f;
  const float c1 = 0x1.63p-1f;       /* 0.693359375 */
  const float c2 = -0x1.bd0106p-13f; /* ln2 - c1 */
  const float t7 = 0x1.a01a02p-13f;  /* 1/5040 */
  const float t6 = 0x1.6c16c2p-10f;  /* 1/720  */
  const float t5 = 0x1.111112p-7f;   /* 1/120  */
  const float t4 = 0x1.555556p-5f;   /* 1/24   */
  const float t3 = 0x1.555556p-3f;   /* 1/6    */
  const float t2 = 0.5f, t1 = 1.0f, t0 = 1.0f;
  if (x < -86.0f) x = -86.0f;
  if (x > 88.0f) x = 88.0f;
  float n = rintf(x * log2e);
  float r = fmaf(-n, c1, x);
  r = fmaf(-n, c2, r);
  float p = t7;
  p = fmaf(p, r, t6);
  p = fmaf(p, r, t5);
  p = fmaf(p, r, t4);
  p = fmaf(p, r, t3);
  p = fmaf(p, r, t2);
  p = fmaf(p, r, t1);
  p = fmaf(p, r, t0);
  int ni = (int)n;
  uint32_t bits = (uint32_t)(ni + 127) << 23;
  float two_n;
  memcpy(&two_n, &bits, sizeof two_n);
  return p * two_n;
}

void ora_spec_exp_n(uint32_t n, const float *x, float *out) {
  for (uint32_t i = 0; i < n; ++i) out[i] = ora_spec_exp(x[i]);
}

/* fp16 bit pattern -> exact double */
double ora_f16_to_f64(uint16_t h) {
  int neg = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int m = h & 1023;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24);
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(m + 1024), e - 25);
  }
  return neg ? -v : v;
}

/* log(1+y) for 0 <= y <= 1, "spec-log1p", defined so that any IEEE-754 fp32
 * machine gets the same bits: z = y/(2+y) (IEEE division), log1p(y) =
 * 2 atanh(z) = 2z (1 + z^2/3 + z^4/5 + ... + z^14/15): the series of atanh in
 * z^2 <= 1/9, coefficients fp32(1/(2n+1)), Horner with fmaf, then (2z) * p.
 * Used by the softplus of the DeepSeek-style scoring sqrt(softplus(l)) ("256
 * experts, 512 lines", section "The constant that always said 256"). */
float ora_spec_log1p(float y) {
  const float c7 = 0x1.111112p-4f; /* 1/15 */
  const float c6 = 0x1.3b13b2p-4f; /* 1/13 */
  const float c5 = 0x1.745d18p-4f; /* 1/11 */
  const float c4 = 0x1.c71c72p-4f; /* 1/9  */
  const float c3 = 0x1.24924ap-3f; /* 1/7  */
  const float c2 = 0x1.99999ap-3f; /* 1/5  */
  const float c1 = 0x1.555556p-2f; /* 1/3  */
  const float c0 = 1.0f;
  const float z = y / (2.0f + y);
  const float z2 = z * z;
  float p = c7;
  p = fmaf(p, z2, c6);
  p = fmaf(p, z2, c5);
  p = fmaf(p, z2, c4);
  p = fmaf(p, z2, c3);
  p = fmaf(p, z2, c2);
  p = fmaf(p, z2, c1);
  p = fmaf(p, z2, c0);
  return (2.0f * z) * p;
}

/* sqrt(softplus(l)) with softplus(l) = max(l, 0) + log1p(e(-|l|)): spec-exp,
 * spec-log1p, IEEE add and sqrt */
float ora_sqrt_softplus(float l) {
  const float m = l > 0.0f ? l : 0.0f;
  const float e = ora_spec_exp(-fabsf(l));
  return sqrtf(m + ora_spec_log1p(e));
}

/* Router logits l[t][e] = sum_i x[t][i] * w_r[e][i] (the router GEMM in front
 * of the scoring: per token, n_expert logits feed the expert scores -- "256
 * experts, 512 lines", "The constant that always said 256").  The pages give
 * no precision or order for it, so the plain definition is taken: every
 * product of the fp32 inputs (exact in double: 24 + 24 significand bits), the
 * products summed in double in ascending i, and the sum rounded once to fp32. */
void ora_router_logits(uint32_t T, uint32_t E, uint32_t d, const float *x, const float *w_r,
                       float *logits) {
  for (uint32_t t = 0; t < T; ++t) {
    for (uint32_t e = 0; e < E; ++e) {
      double sum = 0.0;
      for (uint32_t i = 0; i < d; ++i)
        sum += (double)x[(size_t)t * d + i] * (double)w_r[(size_t)e * d + i];
      logits[(size_t)t * E + e] = (float)sum;
    }
  }
}

/* ------------------------------------------------------------------ A1 score */
void ora_score(uint32_t E, const float *logit, const float *bias, float *sigma, float *c) {
  for (uint32_t i = 0; i < E; ++i) {
    float e = ora_spec_exp(-logit[i]);
    float sg = 1.0f / (1.0f + e);
    if (sigma) sigma[i] = sg;
    c[i] = sg + bias[i];
  }
}

/* per-expert score p_i of scoring function fn (ORA_SCORE_*) and selection score
 * c_i = p_i + b_i */
void ora_score_fn(int32_t fn, uint32_t E, const float *logit, const float *bias, float *p,
                  float *c) {
  if (fn == ORA_SCORE_SIGMOID) {
    ora_score(E, logit, bias, p, c);
    return;
  }
  for (uint32_t i = 0; i < E; ++i) {
    const float v = ora_sqrt_softplus(logit[i]);
    if (p) p[i] = v;
    c[i] = v + bias[i];
  }
}

/* the score in fp64 (routing weights): sigmoid, or sqrt(softplus) in its
 * overflow-free form */
static double score_f64(int32_t fn, double l) {
  if (fn == ORA_SCORE_SIGMOID) return 1.0 / (1.0 + exp(-l));
  return sqrt((l > 0.0 ? l : 0.0) + log1p(exp(-fabs(l))));
}

/* ------------------------------------------------------------------ A2 top-k
 * Slot j takes the largest c among experts not yet taken; scanning upward
 * with a strict '>' keeps the lower index on ties. */
void ora_topk(uint32_t E, uint32_t k, const float *c, int32_t *idx) {
  unsigned char *taken = (unsigned char *)calloc(E, 1);
  for (uint32_t j = 0; j < k; ++j) {
    int32_t best = -1;
    for (uint32_t i = 0; i < E; ++i) {
      if (taken[i]) continue;
      if (best < 0 || c[i] > c[best]) best = (int32_t)i;
    }
    idx[j] = best;
    taken[best] = 1;
  }
  free(taken);
}

/* router for T tokens with scoring function fn; weights w_j = s * p_j / sum_j
 * p_j in fp64 */
void ora_route_fn(int32_t fn, uint32_t T, uint32_t E, uint32_t k, float s, const float *logits,
                  const float *bias, int32_t *idx, float *w) {
  float *c = (float *)malloc(sizeof(float) * E);
  for (uint32_t t = 0; t < T; ++t) {
    const float *l = logits + (size_t)t * E;
    ora_score_fn(fn, E, l, bias, NULL, c);
    ora_topk(E, k, c, idx + (size_t)t * k);
    if (w) {
      double sum = 0.0;
      for (uint32_t j = 0; j < k; ++j) sum += score_f64(fn, (double)l[idx[t * k + j]]);
      for (uint32_t j = 0; j < k; ++j) {
        const double p = score_f64(fn, (double)l[idx[t * k + j]]);
        w[t * k + j] = (float)((double)s * p / sum);
      }
    }
  }
  free(c);
}

/* sigmoid router (the GLM-5.2 / Hy3 scoring) */
void ora_route(uint32_t T, uint32_t E, uint32_t k, float s, const float *logits,
               const float *bias, int32_t *idx, float *w) {
  ora_route_fn(ORA_SCORE_SIGMOID, T, E, k, s, logits, bias, idx, w);
}

/* ------------------------------------------------------------------ A3 permute
 * Counting sort, stable in (token, slot) order. */
void ora_permute(uint32_t T, uint32_t E, uint32_t k, const int32_t *idx, int32_t *off,
                 int32_t *perm, int32_t *pos) {
  uint32_t R = T * k;
  int32_t *cursor = (int32_t *)calloc(E + 1, sizeof(int32_t));
  for (uint32_t e = 0; e <= E; ++e) off[e] = 0;
  for (uint32_t r = 0; r < R; ++r) off[idx[r] + 1] += 1;
  for (uint32_t e = 0; e < E; ++e) off[e + 1] += off[e];
  for (uint32_t e = 0; e < E; ++e) cursor[e] = off[e];
  for (uint32_t r = 0; r < R; ++r) {
    int32_t p = cursor[idx[r]]++;
    if (perm) perm[p] = (int32_t)r;
    if (pos) pos[r] = p;
  }
  free(cursor);
}

/* ------------------------------------------------------------------ A4 quantise */
void ora_quantize(uint32_t n, const float *x, int8_t *q, float *scale) {
  for (uint32_t b = 0; b < n / 32; ++b) {
    const float *xb = x + 32 * b;
    float a = 0.0f;
    for (int i = 0; i < 32; ++i) {
      float v = fabsf(xb[i]);
      if (v > a) a = v;
    }
    float sx = a / 127.0f;
    scale[b] = sx;
    for (int i = 0; i < 32; ++i) {
      if (sx == 0.0f) {
        q[32 * b + i] = 0;
        continue;
      }
      float v = roundf(xb[i] / sx); /* C99 roundf: halfway cases away from zero */
      if (v > 127.0f) v = 127.0f;
      if (v < -127.0f) v = -127.0f;
      q[32 * b + i] = (int8_t)v;
    }
  }
}

/* ------------------------------------------------------------------ A10 2-bit */
void ora_decode_q2(uint32_t K, const uint8_t *codes, int8_t *out) {
  for (uint32_t i = 0; i < K; ++i) {
    int c = (codes[i / 4] >> (2 * (i % 4))) & 3;
    out[i] = (int8_t)(2 * c - 3);
  }
}

/* ------------------------------------------------------------------ 4-bit e2m1 */
/* e2m1 (the OCP microscaling 4-bit float: 1 sign, 2 exponent bits with bias
 * 1, 1 mantissa bit, no infinities or NaN): code c = s e1 e0 m, value
 * (-1)^s * (e == 0 ? m / 2 : 2^(e-1) * (1 + m/2)), i.e. 0, 0.5, 1, 1.5, 2, 3,
 * 4, 6.  Weight i of a row sits at bits 4(i%2) of byte i/2 (low nibble first).
 * Decoded to int8 as TWICE the value (0, 1, 2, 3, 4, 6, 8, 12), so that block
 * dots stay exact integers; the matvec halves the weight scale. */
void ora_decode_e2m1(uint32_t K, const uint8_t *codes, int8_t *out) {
  for (uint32_t i = 0; i < K; ++i) {
    const int c = (codes[i / 2] >> (4 * (i % 2))) & 15;
    const int sgn = c >> 3, e = (c >> 1) & 3, m = c & 1;
    const int twice = e == 0 ? m : (1 << e) + m * (1 << (e - 1)); /* 2 * value */
    out[i] = (int8_t)(sgn ? -twice : twice);
  }
}

/* ------------------------------------------------------------------ A5/A7 dots */
void ora_block_dots(int32_t fmt, uint32_t K, const void *wq_row, const int8_t *xq,
                    int32_t *isum) {
  int8_t *w = (int8_t *)malloc(K);
  if (fmt == ORA_FMT_Q2S)
    ora_decode_q2(K, (const uint8_t *)wq_row, w);
  else if (fmt == ORA_FMT_E2M1)
    ora_decode_e2m1(K, (const uint8_t *)wq_row, w);
  else
    memcpy(w, wq_row, K);
  for (uint32_t b = 0; b < K / 32; ++b) {
    int32_t acc = 0;
    for (int i = 0; i < 32; ++i) acc += (int32_t)w[32 * b + i] * (int32_t)xq[32 * b + i];
    isum[b] = acc;
  }
  free(w);
}

static size_t row_bytes(int32_t fmt, uint32_t K) {
  return fmt == ORA_FMT_Q2S ? K / 4 : fmt == ORA_FMT_E2M1 ? K / 2 : K;
}

void ora_matvec(int32_t fmt, uint32_t rows, uint32_t K, const void *wq, const uint16_t *ws,
                const int8_t *xq, const float *xs, double *out) {
  uint32_t nb = K / 32;
  int32_t *isum = (int32_t *)malloc(sizeof(int32_t) * nb);
  /* e2m1 block dots are of twice the weights: half the scale (exact) */
  const double wmul = fmt == ORA_FMT_E2M1 ? 0.5 : 1.0;
  for (uint32_t n = 0; n < rows; ++n) {
    const char *row = (const char *)wq + (size_t)n * row_bytes(fmt, K);
    ora_block_dots(fmt, K, row, xq, isum);
    double acc = 0.0;
    for (uint32_t b = 0; b < nb; ++b)
      acc += (double)isum[b] *
             (wmul * ora_f16_to_f64(ws[(size_t)n * nb + b]) * (double)xs[b]);
    out[n] = acc;
  }
  free(isum);
}

/* one expert on one quantised activation row: hq/hs (may be NULL) and o[d] */
int ora_expert_row(int32_t fmt, uint32_t d, uint32_t width, const ora_expert *ex,
                   const int8_t *xq, const float *xs, int8_t *hq, float *hs, double *o) {
  if (!ex || !ex->gate_q || !ex->gate_s || !ex->up_q || !ex->up_s || !ex->down_q ||
      !ex->down_s)
    return ORA_MISSING_EXPERT;
  double *g = (double *)malloc(sizeof(double) * width);
  double *u = (double *)malloc(sizeof(double) * width);
  float *h = (float *)malloc(sizeof(float) * width);
  int8_t *hq_l = (int8_t *)malloc(width);
  float *hs_l = (float *)malloc(sizeof(float) * (width / 32));
  ora_matvec(fmt, width, d, ex->gate_q, ex->gate_s, xq, xs, g);
  ora_matvec(fmt, width, d, ex->up_q, ex->up_s, xq, xs, u);
  for (uint32_t n = 0; n < width; ++n) h[n] = (float)(g[n] / (1.0 + exp(-g[n])) * u[n]);
  ora_quantize(width, h, hq_l, hs_l);
  ora_matvec(fmt, d, width, ex->down_q, ex->down_s, hq_l, hs_l, o);
  if (hq) memcpy(hq, hq_l, width);
  if (hs) memcpy(hs, hs_l, sizeof(float) * (width / 32));
  free(g);
  free(u);
  free(h);
  free(hq_l);
  free(hs_l);
  return ORA_OK;
}

/* ------------------------------------------------------------------ the layer */
int ora_layer(const ora_desc *desc, const ora_expert *experts, const ora_expert *shared,
              uint32_t T, const float *x, const float *logits, const float *bias,
              const uint8_t *want, ora_out *out) {
  uint32_t E = desc->n_expert, k = desc->top_k, d = desc->d, f = desc->f, fs = desc->f_shared;
  if (E == 0 || k == 0 || k > E || d == 0 || f == 0 || d % 32 || f % 32 || fs % 32)
    return ORA_BAD_ARG;
  if (desc->routed_fmt != ORA_FMT_Q8_0 && desc->routed_fmt != ORA_FMT_Q2S &&
      desc->routed_fmt != ORA_FMT_E2M1)
    return ORA_BAD_ARG;
  uint32_t R = T * k;
  int rc = ORA_OK;
  int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (R + 1));
  float *w32 = (float *)malloc(sizeof(float) * (R + 1));
  int32_t *off = (int32_t *)malloc(sizeof(int32_t) * (E + 1));
  int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (R + 1));
  int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * (R + 1));
  int8_t *xq = (int8_t *)malloc((size_t)T * d + 1);
  float *xs = (float *)malloc(sizeof(float) * ((size_t)T * d / 32 + 1));
  double *o = (double *)malloc(sizeof(double) * d);
  double *acc = (double *)malloc(sizeof(double) * d);
  double *wd = (double *)malloc(sizeof(double) * k);
  for (uint32_t t = 0; t < T; ++t)
    ora_quantize(d, x + (size_t)t * d, xq + (size_t)t * d, xs + (size_t)t * d / 32);
  ora_route_fn(desc->score_fn, T, E, k, desc->s, logits, bias, idx, w32);
  ora_permute(T, E, k, idx, off, perm, pos);
  for (uint32_t t = 0; t < T && rc == ORA_OK; ++t) {
    if (want && !want[t]) continue;
    const int8_t *xqt = xq + (size_t)t * d;
    const float *xst = xs + (size_t)t * d / 32;
    const float *l = logits + (size_t)t * E;
    /* routing weights in fp64 (the fp32 copy in w32 is only an output) */
    double sum = 0.0;
    for (uint32_t j = 0; j < k; ++j) sum += score_f64(desc->score_fn, (double)l[idx[t * k + j]]);
    for (uint32_t j = 0; j < k; ++j)
      wd[j] = (double)desc->s * score_f64(desc->score_fn, (double)l[idx[t * k + j]]) / sum;
    for (uint32_t m = 0; m < d; ++m) acc[m] = 0.0;
    if (fs > 0) {
      rc = ora_expert_row(ORA_FMT_Q8_0, d, fs, shared, xqt, xst,
                          out->hq_s ? out->hq_s + (size_t)t * fs : NULL,
                          out->hs_s ? out->hs_s + (size_t)t * fs / 32 : NULL, o);
      if (rc != ORA_OK) break;
      for (uint32_t m = 0; m < d; ++m) acc[m] = o[m];
    }
    for (uint32_t j = 0; j < k; ++j) {
      int32_t e = idx[t * k + j];
      size_t p = (size_t)pos[t * k + j];
      rc = ora_expert_row(desc->routed_fmt, d, f, &experts[e], xqt, xst,
                          out->hq_r ? out->hq_r + p * f : NULL,
                          out->hs_r ? out->hs_r + p * f / 32 : NULL, o);
      if (rc != ORA_OK) break;
      for (uint32_t m = 0; m < d; ++m) acc[m] += wd[j] * o[m];
    }
    if (out->y)
      for (uint32_t m = 0; m < d; ++m) out->y[(size_t)t * d + m] = (float)acc[m];
  }
  if (out->idx) memcpy(out->idx, idx, sizeof(int32_t) * R);
  if (out->w) memcpy(out->w, w32, sizeof(float) * R);
  if (out->off) memcpy(out->off, off, sizeof(int32_t) * (E + 1));
  if (out->perm) memcpy(out->perm, perm, sizeof(int32_t) * R);
  if (out->pos) memcpy(out->pos, pos, sizeof(int32_t) * R);
  if (out->xq) memcpy(out->xq, xq, (size_t)T * d);
  if (out->xs) memcpy(out->xs, xs, sizeof(float) * ((size_t)T * d / 32));
  free(idx);
  free(w32);
  free(off);
  free(perm);
  free(pos);
  free(xq);
  free(xs);
  free(o);
  free(acc);
  free(wd);
  return rc;
}
