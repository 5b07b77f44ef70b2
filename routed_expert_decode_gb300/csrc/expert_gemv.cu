// expert_gemv.cu -- dp4a expert FFN for decode and small batches.
//
// Each selected expert's weights are read once per call and applied to all of
// its rows (the union-of-experts read of NeutronStar README, section "MTP
// speculative decoding", and the per-expert indexed FFN of
// DS4_GLM_INDEXED_PER_EXPERT_FFN).  Dot products are int8 x int8 -> int32 per
// 32-block with __dp4a, then scaled by the weight and activation block scales
// (the dp4a expert kernels of "What this branch adds over upstream").
//
// Work items are single output features; a warp streams that feature's gate and
// up rows (Q8_0: one 32-byte load per block per lane, 1 KB per warp
// instruction, no L1 allocation) and dots them with every row of the expert.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerCta = 8;

struct GUArgs {
  const int *plan;
  uint32_t E, k, d, f, fs, R, fmax;
  const int8_t *gq, *uq, *sgq, *suq;
  const uint16_t *gs, *us, *sgs, *sus;
  const int32_t *eslot;  // expert -> weight slot (moe_weights.expert_slot), or null
  const int8_t *xq;  // x codes [T][d]
  const int8_t *xt;  // 2-bit routed weights: x codes, 16-code groups transposed
  const float *xs;
  const int32_t *perm;
  float *h;
  int32_t *tap;
  int routed_fmt;
};

struct DNArgs {
  const int *plan;
  uint32_t E, d, f, fs, R, fmax;
  const int8_t *dq, *sdq;
  const uint16_t *ds, *sds;
  const int32_t *eslot;  // expert -> weight slot (moe_weights.expert_slot), or null
  const int8_t *hq;  // h codes [slots][fmax]
  const int8_t *ht;  // 2-bit routed weights: h codes, 16-code groups transposed
  const float *hs;
  float *o;
  int32_t *tap;
};

// Shape of a warp work item: NF consecutive output features of one expert; a
// pass over 32*J blocks gives lane l the blocks l, l+32, .., l+32(J-1) of each
// of the NF rows of each of the NM matrices, all loaded before any use (32 to
// 64 registers of weight codes in flight per lane, to cover HBM latency with
// 16-24 warps per SM); one plan lookup per item.
// WIDE (gate/up, many tokens): 2 features per item for both formats -- twice the
// codes in flight per warp; it pays when the call streams many experts' rows
// (prefill) and costs a little on small batches, whose items are already few.
template <int FMT, int NM, bool WIDE = false>
__host__ __device__ constexpr int group_nf() {
  return NM == 2 ? (FMT == MOE_FMT_Q2S || WIDE ? 2 : 1) : 4;
}
template <int FMT, int NM, int MAXR>
__host__ __device__ constexpr int group_j() {
  return FMT == MOE_FMT_Q2S && NM == 2 && MAXR < 4 ? 4 : 2;
}

template <int FMT, int MAXR, bool WIDE = false>
__host__ __device__ constexpr int min_ctas() {
  return FMT == MOE_FMT_Q8_0 && MAXR <= 2 && !WIDE ? 3 : 2;
}
// down items are 4 features of a 2048-wide row (one pass each): the 4 rows' codes
// in flight need the registers of 2 CTAs per SM
template <int FMT, int MAXR>
__host__ __device__ constexpr int min_ctas_dn() { return 2; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <bool TAPS>
__device__ __forceinline__ int tap_index(uint32_t n, uint32_t width) {
  if (!TAPS) return -1;
  int jt = -1;
#pragma unroll
  for (int j = kNTap - 1; j >= 0; --j)
    if (tap_feature(j, width) == n) jt = j;
  return jt;
}

// acc[m][f][r] += sum over the K/32 blocks b of
//   dot(codes of row f of matrix m, codes of activation row r) * w-scale * x-scale
// w[m] / ws[m]: first weight row / scale row of the group (rb bytes, nb scales
// a row); activation row r at act + idx[r]*act_stride, its scales at
// act_s + idx[r]*act_s_stride.  tap(m, f, r, b, dot) sees every block dot.
template <int FMT, int NM, int NF, int J, int MAXR, typename Tap>
__device__ __forceinline__ void group_dots(const int8_t *const (&w)[NM],
                                           const uint16_t *const (&ws)[NM], size_t rb,
                                           uint32_t nb, const int8_t *act, size_t act_stride,
                                           const float *act_s, size_t act_s_stride,
                                           const int (&idx)[MAXR], int nr,
                                           float (&acc)[NM][NF][MAXR], Tap tap) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (uint32_t b0 = 0; b0 < nb; b0 += 32 * J) {
    // lanes past the last block load the last block again (valid memory, an
    // L1/L2 hit) and add it with scale 0: no divergent branches, so that the
    // unrolled loads stay in registers
    WBlock<FMT> wb[NM][NF][J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const uint32_t b = min(b0 + lane + 32 * j, nb - 1);
#pragma unroll
      for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int f = 0; f < NF; ++f) wb[m][f][j].load(w[m] + f * rb, b);
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const bool valid = b0 + lane + 32 * j < nb;
      const uint32_t b = min(b0 + lane + 32 * j, nb - 1);
      float sw[NM][NF];
#pragma unroll
      for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int f = 0; f < NF; ++f) {
          sw[m][f] = valid ? half_bits_to_float(ws[m][(size_t)f * nb + b]) * scale_mul<FMT>()
                           : 0.0f;
          wb[m][f][j].prep();
        }
#pragma unroll
      for (int r = 0; r < MAXR; ++r) {
        if (r < nr) {  // warp-uniform
          const W8 x = ld_cached32(act + (size_t)idx[r] * act_stride + 32 * b);
          const float xsc = act_s[(size_t)idx[r] * act_s_stride + b];
          const int sx = WBlock<FMT>::kNeedSum ? block_sum(x) : 0;
#pragma unroll
          for (int m = 0; m < NM; ++m)
#pragma unroll
            for (int f = 0; f < NF; ++f) {
              const int v = wb[m][f][j].dot(x, sx);
              acc[m][f][r] = __fmaf_rn((float)v, sw[m][f] * xsc, acc[m][f][r]);
              if (valid) tap(m, f, r, b, v);
            }
        }
      }
    }
  }
}

// g/u of features [n0, n0 + NF) for rows [row0, row0 + nrows) of one expert;
// h = silu(g)*u.  Rows go in passes of at most MAXR (a later pass re-reads the
// group's rows, which the first pass has just brought into L2).
template <int FMT, int NF, int J, int MAXR, bool TAPS>
__device__ __forceinline__ void gateup_group(const GUArgs &a, const int8_t *gq,
                                             const uint16_t *gs, const int8_t *uq,
                                             const uint16_t *us, uint32_t width, int n0,
                                             int row0, int nrows, bool shared) {
  const int lane = threadIdx.x & 31;
  const uint32_t d = a.d, nb = d / 32;
  const size_t rb = row_bytes(FMT, d);
  const int8_t *const w[2] = {gq + (size_t)n0 * rb, uq + (size_t)n0 * rb};
  const uint16_t *const ws[2] = {gs + (size_t)n0 * nb, us + (size_t)n0 * nb};
  int jt[NF];
#pragma unroll
  for (int f = 0; f < NF; ++f) jt[f] = tap_index<TAPS>((uint32_t)(n0 + f), width);
  for (int r0 = 0; r0 < nrows; r0 += MAXR) {
    const int nr = min(MAXR, nrows - r0);
    int tok[MAXR];
#pragma unroll
    for (int r = 0; r < MAXR; ++r) {
      const int p = row0 + r0 + r;
      tok[r] = r < nr ? (shared ? p - (int)a.R : a.perm[p] / (int)a.k) : 0;
    }
    float acc[2][NF][MAXR];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int f = 0; f < NF; ++f)
#pragma unroll
        for (int r = 0; r < MAXR; ++r) acc[m][f][r] = 0.0f;
    group_dots<FMT, 2, NF, J, MAXR>(
        w, ws, rb, nb, FMT == MOE_FMT_Q2S ? a.xt : a.xq, d, a.xs, nb, tok, nr, acc,
        [&](int m, int f, int r, uint32_t b, int v) {
          if (TAPS && jt[f] >= 0)
            a.tap[(((size_t)(row0 + r0 + r) * 2 + m) * kNTap + jt[f]) * nb + b] = v;
        });
#pragma unroll
    for (int r = 0; r < MAXR; ++r) {
      if (r < nr) {  // warp-uniform
#pragma unroll
        for (int f = 0; f < NF; ++f) {
          const float g = warp_sum(acc[0][f][r]);
          const float u = warp_sum(acc[1][f][r]);
          if (lane == f) {
            const float hv = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, spec_exp(-g))), u);
            a.h[(size_t)(row0 + r0 + r) * a.fmax + n0 + f] = hv;
          }
        }
      }
    }
  }
}

template <int FMT, int MAXR, bool TAPS, bool WIDE>
__global__ void __launch_bounds__(kWarpsPerCta * 32, (min_ctas<FMT, MAXR, WIDE>()))
    k_gateup(const GUArgs a) {
  pdl_trigger();
  pdl_wait();
  constexpr int NF = group_nf<FMT, 2, WIDE>(), J = group_j<FMT, 2, MAXR>();
  constexpr int NFS = group_nf<MOE_FMT_Q8_0, 2, WIDE>(), JS = group_j<MOE_FMT_Q8_0, 2, MAXR>();
  static_assert(NF % NFS == 0, "the shared expert's groups must tile the routed ones");
  extern __shared__ int gsm[];
  PlanView P(const_cast<int *>(a.plan), a.E);
  const SmemPlan S(gsm, P, a.E);
  const int U = P.hdr[0];
  const int groups = P.hdr[1] / NF;  // every width is a multiple of 32
  const int nwarps = gridDim.x * kWarpsPerCta;
  for (int g = blockIdx.x * kWarpsPerCta + threadIdx.x / 32; g < groups; g += nwarps) {
    const int item = g * NF;
    const int u = find_slot(S.item, U, item);
    const int e = S.e[u];
    const int n0 = item - S.item[u];
    const int row0 = S.row0[u], nrows = S.rows[u];
    if ((uint32_t)e == a.E) {
#pragma unroll 1
      for (int f = 0; f < NF; f += NFS)
        gateup_group<MOE_FMT_Q8_0, NFS, JS, MAXR, TAPS>(a, a.sgq, a.sgs, a.suq, a.sus, a.fs,
                                                        n0 + f, row0, nrows, true);
    } else {
      const size_t we = (size_t)weight_slot(a.eslot, e);  // validated by k_plan
      const size_t qoff = we * a.f * row_bytes(FMT, a.d);
      const size_t soff = we * a.f * (a.d / 32);
      gateup_group<FMT, NF, J, MAXR, TAPS>(a, a.gq + qoff, a.gs + soff, a.uq + qoff,
                                           a.us + soff, a.f, n0, row0, nrows, false);
    }
  }
}

// 16-code groups of a 32-code block transposed as 4x4 bytes: code 16g + 4j + i
// moves to byte 16g + 4i + j (the order the 2-bit block dot consumes)
__device__ __forceinline__ int transposed_lane(int lane) {
  return (lane & 16) | ((lane & 3) << 2) | ((lane >> 2) & 3);
}

// requantise h per 32-block.  A warp unit is 4 consecutive blocks of one slot
// (lane l holds h[4l .. 4l+3] of the 128, so lanes 8j .. 8j+7 hold block j);
// a fixed grid of warps walks the units two at a time, both units' loads
// issued first.  Per block: amax over its 32 values (one 8-lane max over the
// |h| bit patterns), scale amax / 127, codes as quant_one.
__device__ __forceinline__ float4 requant_load(const float *h, uint64_t u, uint32_t groups,
                                               uint32_t fmax, uint32_t R, uint32_t f, uint32_t fs,
                                               uint64_t units, int lane) {
  if (u >= units) return make_float4(0.f, 0.f, 0.f, 0.f);
  const uint32_t slot = (uint32_t)(u / groups), b = (uint32_t)(u % groups) * 4 + (lane >> 3);
  const uint32_t width = slot < R ? f : fs;
  if (32 * b >= width) return make_float4(0.f, 0.f, 0.f, 0.f);
  return *reinterpret_cast<const float4 *>(h + (size_t)slot * fmax + 32 * b + 4 * (lane & 7));
}

__device__ __forceinline__ void requant_store(float4 v, uint64_t u, uint32_t groups,
                                              uint32_t fmax, uint32_t R, uint32_t f, uint32_t fs,
                                              uint64_t units, int lane, int8_t *__restrict__ hq,
                                              float *__restrict__ hs, int8_t *__restrict__ ht) {
  // every lane takes part in the shuffles; out-of-range lanes hold zeros
  uint32_t m = max(max(__float_as_uint(fabsf(v.x)), __float_as_uint(fabsf(v.y))),
                   max(__float_as_uint(fabsf(v.z)), __float_as_uint(fabsf(v.w))));
#pragma unroll
  for (int o = 4; o >= 1; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (u >= units) return;
  const uint32_t slot = (uint32_t)(u / groups), b = (uint32_t)(u % groups) * 4 + (lane >> 3);
  const uint32_t width = slot < R ? f : fs;
  if (32 * b >= width) return;
  const float sc = __fdiv_rn(__uint_as_float(m), 127.0f);
  const int q0 = quant_one(v.x, sc), q1 = quant_one(v.y, sc), q2 = quant_one(v.z, sc),
            q3 = quant_one(v.w, sc);
  const size_t i = (size_t)slot * fmax + 32 * b + 4 * (lane & 7);
  *reinterpret_cast<char4 *>(hq + i) = make_char4((signed char)q0, (signed char)q1,
                                                  (signed char)q2, (signed char)q3);
  if (ht && slot < R) {
    int8_t *tb = ht + (size_t)slot * fmax + 32 * b;
    const int e0 = 4 * (lane & 7);
    tb[transposed_lane(e0)] = (int8_t)q0;
    tb[transposed_lane(e0 + 1)] = (int8_t)q1;
    tb[transposed_lane(e0 + 2)] = (int8_t)q2;
    tb[transposed_lane(e0 + 3)] = (int8_t)q3;
  }
  if ((lane & 7) == 0) hs[(size_t)slot * (fmax / 32) + b] = sc;
}

__global__ void __launch_bounds__(256)
    k_requant(const float *__restrict__ h, uint32_t slots, uint32_t R, uint32_t f, uint32_t fs,
              uint32_t fmax, int8_t *__restrict__ hq, float *__restrict__ hs,
              int8_t *__restrict__ ht) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const uint32_t groups = (fmax + 127) / 128;
  const uint64_t units = (uint64_t)slots * groups;
  const uint64_t nw = (uint64_t)gridDim.x * 8;
  for (uint64_t u = (uint64_t)blockIdx.x * 8 + threadIdx.x / 32; u < units; u += 2 * nw) {
    const float4 v0 = requant_load(h, u, groups, fmax, R, f, fs, units, lane);
    const float4 v1 = requant_load(h, u + nw, groups, fmax, R, f, fs, units, lane);
    requant_store(v0, u, groups, fmax, R, f, fs, units, lane, hq, hs, ht);
    requant_store(v1, u + nw, groups, fmax, R, f, fs, units, lane, hq, hs, ht);
  }
}

// o[slot][m] for m in [m0, m0 + NF), rows of one expert: down rows (K = width)
// against the h codes
template <int FMT, int NF, int J, int MAXR, bool TAPS>
__device__ __forceinline__ void down_group(const DNArgs &a, const int8_t *dq, const uint16_t *ds,
                                           uint32_t width, int m0, int row0, int nrows) {
  const int lane = threadIdx.x & 31;
  const uint32_t nb = width / 32, nbmax = a.fmax / 32;
  const size_t rb = row_bytes(FMT, width);
  const int8_t *const w[1] = {dq + (size_t)m0 * rb};
  const uint16_t *const ws[1] = {ds + (size_t)m0 * nb};
  int jt[NF];
#pragma unroll
  for (int f = 0; f < NF; ++f) jt[f] = tap_index<TAPS>((uint32_t)(m0 + f), a.d);
  for (int r0 = 0; r0 < nrows; r0 += MAXR) {
    const int nr = min(MAXR, nrows - r0);
    int slot[MAXR];
#pragma unroll
    for (int r = 0; r < MAXR; ++r) slot[r] = r < nr ? row0 + r0 + r : row0;
    float acc[1][NF][MAXR];
#pragma unroll
    for (int f = 0; f < NF; ++f)
#pragma unroll
      for (int r = 0; r < MAXR; ++r) acc[0][f][r] = 0.0f;
    group_dots<FMT, 1, NF, J, MAXR>(
        w, ws, rb, nb, FMT == MOE_FMT_Q2S ? a.ht : a.hq, a.fmax, a.hs, nbmax, slot, nr, acc,
        [&](int, int f, int r, uint32_t b, int v) {
          if (TAPS && jt[f] >= 0) a.tap[((size_t)slot[r] * kNTap + jt[f]) * nbmax + b] = v;
        });
#pragma unroll
    for (int r = 0; r < MAXR; ++r) {
      if (r < nr) {  // warp-uniform
#pragma unroll
        for (int f = 0; f < NF; ++f) {
          const float v = warp_sum(acc[0][f][r]);
          if (lane == f) a.o[(size_t)slot[r] * a.d + m0 + f] = v;
        }
      }
    }
  }
}

template <int FMT, int MAXR, bool TAPS>
__global__ void __launch_bounds__(kWarpsPerCta * 32, (min_ctas_dn<FMT, MAXR>())) k_down(const DNArgs a) {
  pdl_trigger();
  pdl_wait();
  constexpr int NF = group_nf<FMT, 1>(), J = group_j<FMT, 1, MAXR>();
  constexpr int NFS = group_nf<MOE_FMT_Q8_0, 1>(), JS = group_j<MOE_FMT_Q8_0, 1, MAXR>();
  static_assert(NF % NFS == 0, "the shared expert's groups must tile the routed ones");
  extern __shared__ int gsm[];
  PlanView P(const_cast<int *>(a.plan), a.E);
  const SmemPlan S(gsm, P, a.E);
  const int per = (int)a.d / NF;  // groups per expert
  const int groups = P.hdr[2] / NF;
  const int nwarps = gridDim.x * kWarpsPerCta;
  for (int g = blockIdx.x * kWarpsPerCta + threadIdx.x / 32; g < groups; g += nwarps) {
    const int u = g / per;
    const int m0 = (g - u * per) * NF;
    const int e = S.e[u];
    const int row0 = S.row0[u], nrows = S.rows[u];
    if ((uint32_t)e == a.E) {
#pragma unroll 1
      for (int f = 0; f < NF; f += NFS)
        down_group<MOE_FMT_Q8_0, NFS, JS, MAXR, TAPS>(a, a.sdq, a.sds, a.fs, m0 + f, row0, nrows);
    } else {
      const size_t we = (size_t)weight_slot(a.eslot, e);  // validated by k_plan
      const size_t qoff = we * a.d * row_bytes(FMT, a.f);
      const size_t soff = we * a.d * (a.f / 32);
      down_group<FMT, NF, J, MAXR, TAPS>(a, a.dq + qoff, a.ds + soff, a.f, m0, row0, nrows);
    }
  }
}

// y[t][m] = o_shared[t][m] + sum_j w[t,j] * o[pos[t,j]][m], in that order
// (only the slots of experts in [e_lo, e_hi), and the shared term if `shared`:
// an expert-parallel rank's share of the sum).  A thread takes 4 consecutive m
// of one token (d is a multiple of 32) and issues the loads of 8 terms before
// their multiply-adds.
__global__ void __launch_bounds__(256)
    k_combine(const float *__restrict__ o, const float *__restrict__ w,
              const int32_t *__restrict__ pos, const int32_t *__restrict__ idx, uint32_t T,
              uint32_t k, uint32_t d, uint32_t R, bool shared, uint32_t e_lo, uint32_t e_hi,
              bool all_experts, const int *__restrict__ plan, float *__restrict__ y) {
  pdl_trigger();
  pdl_wait();
  const uint32_t d4 = d / 4;
  const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (uint64_t)T * d4) return;
  const uint32_t t = (uint32_t)(i / d4), m = 4 * (uint32_t)(i % d4);
  float *yo = y + (size_t)t * d + m;
  // y is the caller's: 16-byte stores only where it is 16-byte aligned
  auto store = [&](float4 v) {
    if (((uintptr_t)y & 15u) == 0) {
      *reinterpret_cast<float4 *>(yo) = v;
    } else {
      yo[0] = v.x;
      yo[1] = v.y;
      yo[2] = v.z;
      yo[3] = v.w;
    }
  };
  if (plan[4] != 1) {  // rejected routing arrays: no expert ran, pos[] is not trusted
    store(make_float4(0.0f, 0.0f, 0.0f, 0.0f));
    return;
  }
  float4 acc = shared ? *reinterpret_cast<const float4 *>(o + ((size_t)R + t) * d + m)
                      : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (uint32_t j0 = 0; j0 < k; j0 += 8) {
    float4 ov[8];
    float wv[8];
    bool use[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const uint32_t j = j0 + (uint32_t)jj;
      use[jj] = j < k;
      if (use[jj] && !all_experts) {
        const uint32_t e = (uint32_t)idx[(size_t)t * k + j];
        use[jj] = e >= e_lo && e < e_hi;
      }
      if (use[jj]) {
        const int p = pos[(size_t)t * k + j];
        wv[jj] = w[(size_t)t * k + j];
        ov[jj] = *reinterpret_cast<const float4 *>(o + (size_t)p * d + m);
      }
    }
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      if (use[jj]) {
        acc.x = __fmaf_rn(wv[jj], ov[jj].x, acc.x);
        acc.y = __fmaf_rn(wv[jj], ov[jj].y, acc.y);
        acc.z = __fmaf_rn(wv[jj], ov[jj].z, acc.z);
        acc.w = __fmaf_rn(wv[jj], ov[jj].w, acc.w);
      }
    }
  }
  store(acc);
}

// resident CTAs per SM of a persistent GEMV kernel with `smem` dynamic bytes
template <typename K>
cudaError_t grid_for(K kernel, size_t smem, bool &big_smem, int &per_sm) {
  if (smem > 48 * 1024 && !big_smem) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    big_smem = true;
  }
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kWarpsPerCta * 32, smem) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return cudaSuccess;
}

template <int FMT, int MAXR, bool TAPS, bool WIDE>
cudaError_t run_gateup(const Ctx &c, const GUArgs &a) {
  static bool big_smem = false;
  auto kern = k_gateup<FMT, MAXR, TAPS, WIDE>;
  const size_t smem = smem_plan_bytes(c.desc.n_expert);
  int per_sm = 1;
  cudaError_t e = grid_for(kern, smem, big_smem, per_sm);
  if (e != cudaSuccess) return e;
  e = launch_k(kern, per_sm * c.sm_count, kWarpsPerCta * 32, smem, c.stream, c.chained, a);
  c.chained = true;
  return e;
}

template <int FMT, int MAXR, bool TAPS>
cudaError_t run_down(const Ctx &c, const DNArgs &a) {
  static bool big_smem = false;
  auto kern = k_down<FMT, MAXR, TAPS>;
  const size_t smem = smem_plan_bytes(c.desc.n_expert);
  int per_sm = 1;
  cudaError_t e = grid_for(kern, smem, big_smem, per_sm);
  if (e != cudaSuccess) return e;
  e = launch_k(kern, per_sm * c.sm_count, kWarpsPerCta * 32, smem, c.stream, c.chained, a);
  c.chained = true;
  return e;
}

// rows per pass: an expert has at most T rows; more than 4 take several passes
int maxr_for(uint32_t T) { return T <= 1 ? 1 : T <= 2 ? 2 : 4; }
// tokens per call from which the gate/up items are 2 features wide (gate/up
// GEMV on the 256-expert layer, 1 -> 2 features: T=16 401 -> 426 us, T=32
// 481 -> 446, T=64 713 -> 637, T=128 807 -> 700, T=512 598 -> 512)
constexpr uint32_t kWideGateupT = 32;

template <int FMT, int MAXR, bool WIDE = false>
cudaError_t gu_taps(const Ctx &c, const GUArgs &a, bool taps) {
  return taps ? run_gateup<FMT, MAXR, true, WIDE>(c, a) : run_gateup<FMT, MAXR, false, WIDE>(c, a);
}
template <int FMT, int MAXR>
cudaError_t dn_taps(const Ctx &c, const DNArgs &a, bool taps) {
  return taps ? run_down<FMT, MAXR, true>(c, a) : run_down<FMT, MAXR, false>(c, a);
}

template <int FMT>
cudaError_t gu_maxr(const Ctx &c, const GUArgs &a, bool taps) {
  switch (maxr_for(c.T)) {
    case 1: return gu_taps<FMT, 1>(c, a, taps);
    case 2: return gu_taps<FMT, 2>(c, a, taps);
    default:
      return c.T >= kWideGateupT ? gu_taps<FMT, 4, true>(c, a, taps) : gu_taps<FMT, 4>(c, a, taps);
  }
}
template <int FMT>
cudaError_t dn_maxr(const Ctx &c, const DNArgs &a, bool taps) {
  switch (maxr_for(c.T)) {
    case 1: return dn_taps<FMT, 1>(c, a, taps);
    case 2: return dn_taps<FMT, 2>(c, a, taps);
    default: return dn_taps<FMT, 4>(c, a, taps);
  }
}

}  // namespace

cudaError_t launch_gateup(const Ctx &c, const int32_t *perm) {
  if (c.T == 0) return cudaSuccess;
  if (stream_gateup_ok(c)) return launch_gateup_stream(c, perm);
  GUArgs a;
  a.plan = (const int *)(c.ws + c.L.plan);
  a.E = c.desc.n_expert;
  a.k = c.desc.top_k;
  a.d = c.desc.d;
  a.f = c.desc.f;
  a.fs = c.desc.f_shared;
  a.R = c.R;
  a.fmax = c.fmax;
  a.gq = (const int8_t *)c.wts.gate.q;
  a.uq = (const int8_t *)c.wts.up.q;
  a.gs = c.wts.gate.scale;
  a.us = c.wts.up.scale;
  a.sgq = (const int8_t *)c.wts.s_gate.q;
  a.suq = (const int8_t *)c.wts.s_up.q;
  a.sgs = c.wts.s_gate.scale;
  a.sus = c.wts.s_up.scale;
  a.eslot = c.wts.expert_slot;
  a.xq = (const int8_t *)(c.ws + c.L.xq);
  a.xt = c.L.xt ? (const int8_t *)(c.ws + c.L.xt) : nullptr;
  a.xs = (const float *)(c.ws + c.L.xs);
  a.perm = perm;
  a.h = (float *)(c.ws + c.L.h);
  a.tap = (int32_t *)(c.ws + c.L.tap_gu);
  a.routed_fmt = c.desc.routed_fmt;
  const bool taps = (c.desc.flags & MOE_FLAG_DEBUG_TAPS) != 0;
  switch (c.desc.routed_fmt) {
    case MOE_FMT_Q2S: return gu_maxr<MOE_FMT_Q2S>(c, a, taps);
    case MOE_FMT_E2M1: return gu_maxr<MOE_FMT_E2M1>(c, a, taps);
    default: return gu_maxr<MOE_FMT_Q8_0>(c, a, taps);
  }
}

cudaError_t launch_requant_h(const Ctx &c) {
  const uint32_t slots = c.R + (c.desc.f_shared ? c.T : 0);
  const uint64_t units = (uint64_t)slots * ((c.fmax + 127) / 128);
  if (units == 0) return cudaSuccess;
  // a fixed grid (6 CTAs of 8 warps an SM: all resident at the kernel's 40
  // registers a thread) walking the units, two a warp at a time
  const uint64_t ctas = std::min<uint64_t>((units + 15) / 16, (uint64_t)c.sm_count * 6);
  const cudaError_t e = launch_k(
      k_requant, (unsigned)ctas, 256, 0, c.stream, c.chained,
      (const float *)(c.ws + c.L.h), slots, c.R, c.desc.f, c.desc.f_shared, c.fmax,
      (int8_t *)(c.ws + c.L.hq), (float *)(c.ws + c.L.hs),
      c.L.ht ? (int8_t *)(c.ws + c.L.ht) : nullptr);
  c.chained = true;
  return e;
}

cudaError_t launch_down(const Ctx &c) {
  if (c.T == 0) return cudaSuccess;
  if (stream_down_ok(c)) return launch_down_stream(c);
  DNArgs a;
  a.plan = (const int *)(c.ws + c.L.plan);
  a.E = c.desc.n_expert;
  a.d = c.desc.d;
  a.f = c.desc.f;
  a.fs = c.desc.f_shared;
  a.R = c.R;
  a.fmax = c.fmax;
  a.dq = (const int8_t *)c.wts.down.q;
  a.ds = c.wts.down.scale;
  a.eslot = c.wts.expert_slot;
  a.sdq = (const int8_t *)c.wts.s_down.q;
  a.sds = c.wts.s_down.scale;
  a.hq = (const int8_t *)(c.ws + c.L.hq);
  a.ht = c.L.ht ? (const int8_t *)(c.ws + c.L.ht) : nullptr;
  a.hs = (const float *)(c.ws + c.L.hs);
  a.o = (float *)(c.ws + c.L.o);
  a.tap = (int32_t *)(c.ws + c.L.tap_dn);
  const bool taps = (c.desc.flags & MOE_FLAG_DEBUG_TAPS) != 0;
  switch (c.desc.routed_fmt) {
    case MOE_FMT_Q2S: return dn_maxr<MOE_FMT_Q2S>(c, a, taps);
    case MOE_FMT_E2M1: return dn_maxr<MOE_FMT_E2M1>(c, a, taps);
    default: return dn_maxr<MOE_FMT_Q8_0>(c, a, taps);
  }
}

cudaError_t launch_combine(const Ctx &c, const float *w, const int32_t *pos,
                           const int32_t *idx, float *y) {
  const uint64_t n = (uint64_t)c.T * (c.desc.d / 4);  // threads: 4 outputs each
  if (n == 0) return cudaSuccess;
  const bool all = c.e_lo == 0 && c.e_hi >= c.desc.n_expert;
  const cudaError_t e = launch_k(
      k_combine, (unsigned)((n + 255) / 256), 256, 0, c.stream, c.chained,
      (const float *)(c.ws + c.L.o), w, pos, idx, c.T, c.desc.top_k, c.desc.d, c.R,
      c.desc.f_shared > 0 && c.shared_on, c.e_lo, c.e_hi, all, (const int *)(c.ws + c.L.plan),
      y);
  c.chained = true;
  return e;
}

}  // namespace moe
