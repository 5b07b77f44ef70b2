/*
 * oracle.h -- plain, slow CPU oracle of the routed-MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * bench's CPU-baseline leg may load this library.  It shares no code, header,
 * table or constant with the CUDA library, and neither includes the other.
 *
 * What it computes (the layer the pages describe, stated in full):
 *  - score    : sigma_i = 1/(1+e(-l_i)), c_i = sigma_i + b_i, in fp32, where e()
 *               is "spec-exp" (ora_spec_exp below).  Sigmoid routing with an
 *               expert-selection bias, top-8: "256 experts, 512 lines", section
 *               "Why GLM-5.2 in an engine built for DeepSeek"; NeutronStar main
 *               README, Hy3 paragraph ("192-expert top-8 sigmoid router with
 *               expert bias").
 *  - DeepSeek : p_i = sqrt(softplus(l_i)) in place of sigma_i (spec-log1p below),
 *               top-6, scale 1.5, E = 384 ("256 experts, 512 lines", section
 *               "The constant that always said 256").
 *  - router   : logits l = x . W_r^T: exact products of the fp32 inputs summed
 *               in fp64, rounded once to fp32 (ora_router_logits; the pages give
 *               no precision or order for the router GEMM).
 *  - top-k    : k indices of largest c; equal c -> lower index first; slots in
 *               order of c descending.  Weight w_j = s * sigma_j / sum_j sigma_j
 *               (fp64).  The parameterised n_expert/top_k/scale router:
 *               "256 experts, 512 lines", section "The constant that always
 *               said 256".
 *  - permute  : stable counting sort of the T*k (token, slot) rows by expert:
 *               off[E+1], perm[R], pos[R].  Per-expert batches: NeutronStar
 *               README, sections "MTP speculative decoding" (indexed per-expert
 *               FFN, union expert loads) and "Long-prompt prefill".
 *  - quantise : per 32-block, a = max|x|, sx = a/127 (fp32), q = clamp(
 *               round_half_away(x/sx), -127, 127); sx == 0 gives q = 0.  One
 *               recipe for every path (NeutronStar main README, Hy3 chunked
 *               prefill paragraph: batch kernels that quantised on a different
 *               path flipped near-tie picks).
 *  - expert   : g_n = sum_b isum_b(Wg[n], xq) * wsg[n][b] * xs[b] with isum_b an
 *               exact int32 dot of 32 int8 pairs (the dp4a technique: NeutronStar
 *               README, "What this branch adds over upstream"); same for u;
 *               h = g/(1+exp(-g))*u in fp64 (libm exp); h rounded to fp32 and
 *               requantised as above;
 *               o_m = sum_b isum_b(Wd[m], hq) * wsd[m][b] * hs[b].  fp64 sums in
 *               block order.  Q8_0 weights ("everything that makes decisions
 *               stays at Q8_0/F32": NeutronStar README, "The model").
 *  - 2-bit    : code c of weight i sits at bits 2(i%4) of byte i/4 (LSB
 *               first) and means the int8 value 2c-3.
 *  - combine  : y[t] = o_shared[t] + sum_{j<k} w[t,j] * o[(t,j)] in that order
 *               (fp64, then rounded to fp32).  Shared expert: "MoE with shared
 *               expert", "256 experts, 512 lines", section "Why GLM-5.2 ...".
 * NaN or infinite inputs are unsupported.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

enum { ORA_FMT_Q8_0 = 0, ORA_FMT_Q2S = 1, ORA_FMT_E2M1 = 2 };
/* scoring of a logit: sigmoid (GLM-5.2, Hy3) or sqrt(softplus) (DeepSeek) */
enum { ORA_SCORE_SIGMOID = 0, ORA_SCORE_SQRT_SOFTPLUS = 1 };
enum { ORA_OK = 0, ORA_BAD_ARG = 1, ORA_MISSING_EXPERT = 2, ORA_NO_MEMORY = 3 };

/* One expert's weights, planar: code plane + fp16 scale plane (bit patterns).
 * gate/up: [width][d] (Q2S: [width][d/4] bytes, E2M1: [width][d/2] bytes),
 * scales [width][d/32]; down: [d][width] (Q2S: [d][width/4], E2M1:
 * [d][width/2]), scales [d][width/32]. */
typedef struct {
  const void *gate_q;
  const uint16_t *gate_s;
  const void *up_q;
  const uint16_t *up_s;
  const void *down_q;
  const uint16_t *down_s;
} ora_expert;

typedef struct {
  uint32_t n_expert, top_k, d, f, f_shared; /* f_shared == 0: no shared expert */
  int32_t routed_fmt;                       /* ORA_FMT_Q8_0, ORA_FMT_Q2S or ORA_FMT_E2M1 */
  float s;                                  /* routing scale */
  int32_t score_fn;                         /* ORA_SCORE_* */
} ora_desc;

/* Outputs of ora_layer; any pointer may be NULL.
 * Routed hidden rows hq_r/hs_r are stored at their permuted position p = pos[t*k+j];
 * shared rows hq_s/hs_s at token t. */
typedef struct {
  int32_t *idx;  /* [T*k] */
  float *w;      /* [T*k] */
  int32_t *off;  /* [E+1] */
  int32_t *perm; /* [T*k] */
  int32_t *pos;  /* [T*k] */
  int8_t *xq;    /* [T*d] */
  float *xs;     /* [T*d/32] */
  int8_t *hq_r;  /* [T*k*f] */
  float *hs_r;   /* [T*k*f/32] */
  int8_t *hq_s;  /* [T*f_shared] */
  float *hs_s;   /* [T*f_shared/32] */
  float *y;      /* [T*d] */
} ora_out;

float ora_spec_exp(float x);
void ora_spec_exp_n(uint32_t n, const float *x, float *out);
double ora_f16_to_f64(uint16_t h);
float ora_spec_log1p(float y);
float ora_sqrt_softplus(float l);
void ora_router_logits(uint32_t T, uint32_t E, uint32_t d, const float *x, const float *w_r,
                       float *logits);
void ora_score(uint32_t E, const float *logit, const float *bias, float *sigma, float *c);
void ora_score_fn(int32_t fn, uint32_t E, const float *logit, const float *bias, float *p,
                  float *c);
void ora_route_fn(int32_t fn, uint32_t T, uint32_t E, uint32_t k, float s, const float *logits,
                  const float *bias, int32_t *idx, float *w);
void ora_topk(uint32_t E, uint32_t k, const float *c, int32_t *idx);
void ora_route(uint32_t T, uint32_t E, uint32_t k, float s, const float *logits,
               const float *bias, int32_t *idx, float *w);
void ora_permute(uint32_t T, uint32_t E, uint32_t k, const int32_t *idx, int32_t *off,
                 int32_t *perm, int32_t *pos);
void ora_quantize(uint32_t n, const float *x, int8_t *q, float *scale);
void ora_decode_q2(uint32_t K, const uint8_t *codes, int8_t *out);
void ora_decode_e2m1(uint32_t K, const uint8_t *codes, int8_t *out);
void ora_block_dots(int32_t fmt, uint32_t K, const void *wq_row, const int8_t *xq,
                    int32_t *isum);
void ora_matvec(int32_t fmt, uint32_t rows, uint32_t K, const void *wq, const uint16_t *ws,
                const int8_t *xq, const float *xs, double *out);
int ora_expert_row(int32_t fmt, uint32_t d, uint32_t width, const ora_expert *ex,
                   const int8_t *xq, const float *xs, int8_t *hq, float *hs, double *o);
/* want: [T] flags, NULL = every token.  Routing, permutation and x quantisation
 * always cover all T tokens; expert rows and y only the wanted ones. */
int ora_layer(const ora_desc *desc, const ora_expert *experts, const ora_expert *shared,
              uint32_t T, const float *x, const float *logits, const float *bias,
              const uint8_t *want, ora_out *out);

#ifdef __cplusplus
}
#endif
#endif
