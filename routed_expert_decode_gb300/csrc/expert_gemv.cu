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
  const int8_t *xq;
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
  const int8_t *hq;
  const float *hs;
  float *o;
  int32_t *tap;
};

__device__ __forceinline__ int find_slot(const int *prefix, int U, int item) {
  int lo = 0, hi = U;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid;
  }
  return lo;
}

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

// g/u of feature n for rows [row0, row0 + nrows) of one expert; h = silu(g)*u
template <int FMT, int MAXR, bool TAPS>
__device__ __forceinline__ void gateup_feature(const GUArgs &a, const int8_t *gq,
                                               const uint16_t *gs, const int8_t *uq,
                                               const uint16_t *us, uint32_t width, int n,
                                               int row0, int nrows, bool shared) {
  const int lane = threadIdx.x & 31;
  const uint32_t d = a.d, nb = d / 32;
  const size_t rb = row_bytes(FMT, d);
  const int8_t *grow = gq + (size_t)n * rb;
  const int8_t *urow = uq + (size_t)n * rb;
  const uint16_t *gsr = gs + (size_t)n * nb;
  const uint16_t *usr = us + (size_t)n * nb;
  const int jt = tap_index<TAPS>((uint32_t)n, width);
  for (int r0 = 0; r0 < nrows; r0 += MAXR) {
    const int nr = min(MAXR, nrows - r0);
    int tok[MAXR];
#pragma unroll
    for (int r = 0; r < MAXR; ++r) {
      const int p = row0 + r0 + r;
      tok[r] = r < nr ? (shared ? p - (int)a.R : a.perm[p] / (int)a.k) : 0;
    }
    float accg[MAXR], accu[MAXR];
#pragma unroll
    for (int r = 0; r < MAXR; ++r) accg[r] = accu[r] = 0.0f;
#pragma unroll 2
    for (uint32_t b = lane; b < nb; b += 32) {
      WBlock<FMT> wg, wu;
      wg.load(grow, b);
      wu.load(urow, b);
      const float sg = half_bits_to_float(gsr[b]);
      const float su = half_bits_to_float(usr[b]);
#pragma unroll
      for (int r = 0; r < MAXR; ++r) {
        if (r < nr) {
          const W8 x = ld_cached32(a.xq + (size_t)tok[r] * d + 32 * b);
          const float xsc = a.xs[(size_t)tok[r] * nb + b];
          const int ig = wg.dot(x);
          const int iu = wu.dot(x);
          accg[r] = __fmaf_rn((float)ig, sg * xsc, accg[r]);
          accu[r] = __fmaf_rn((float)iu, su * xsc, accu[r]);
          if (TAPS && jt >= 0) {
            int32_t *tp = a.tap + ((size_t)(row0 + r0 + r) * 2 * kNTap + jt) * nb;
            tp[b] = ig;
            tp[(size_t)kNTap * nb + b] = iu;
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < MAXR; ++r) {
      const float g = warp_sum(accg[r]);
      const float u = warp_sum(accu[r]);
      if (lane == 0 && r < nr) {
        const float hv = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, spec_exp(-g))), u);
        a.h[(size_t)(row0 + r0 + r) * a.fmax + n] = hv;
      }
    }
  }
}

template <int FMT, int MAXR, bool TAPS>
__global__ void __launch_bounds__(kWarpsPerCta * 32, MAXR <= 2 ? 3 : 2) k_gateup(const GUArgs a) {
  PlanView P(const_cast<int *>(a.plan), a.E);
  const int U = P.hdr[0];
  const int total = P.hdr[1];
  const int nwarps = gridDim.x * kWarpsPerCta;
  for (int item = blockIdx.x * kWarpsPerCta + threadIdx.x / 32; item < total; item += nwarps) {
    const int u = find_slot(P.item_gu, U, item);
    const int e = P.act_e[u];
    const int n = item - P.item_gu[u];
    const int row0 = P.act_row0[u], nrows = P.act_rows[u];
    if ((uint32_t)e == a.E) {
      gateup_feature<MOE_FMT_Q8_0, MAXR, TAPS>(a, a.sgq, a.sgs, a.suq, a.sus, a.fs, n, row0,
                                               nrows, true);
    } else {
      const size_t qoff = (size_t)e * a.f * row_bytes(FMT, a.d);
      const size_t soff = (size_t)e * a.f * (a.d / 32);
      gateup_feature<FMT, MAXR, TAPS>(a, a.gq + qoff, a.gs + soff, a.uq + qoff, a.us + soff,
                                      a.f, n, row0, nrows, false);
    }
  }
}

// requantise h per 32-block: one warp per (slot, block)
__global__ void __launch_bounds__(256)
    k_requant(const float *__restrict__ h, uint32_t slots, uint32_t R, uint32_t f, uint32_t fs,
              uint32_t fmax, int8_t *__restrict__ hq, float *__restrict__ hs) {
  const int lane = threadIdx.x & 31;
  const uint32_t nbmax = fmax / 32;
  const uint64_t gw = (uint64_t)blockIdx.x * 8 + threadIdx.x / 32;
  if (gw >= (uint64_t)slots * nbmax) return;
  const uint32_t slot = (uint32_t)(gw / nbmax), b = (uint32_t)(gw % nbmax);
  const uint32_t width = slot < R ? f : fs;
  if (b >= width / 32) return;
  const size_t i = (size_t)slot * fmax + 32 * b + lane;
  const float v = h[i];
  float amax = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = __fdiv_rn(amax, 127.0f);
  hq[i] = (int8_t)quant_one(v, sc);
  if (lane == 0) hs[(size_t)slot * nbmax + b] = sc;
}

// o[slot][m] for rows of one expert: the down row m (K = width) against hq
template <int FMT, int MAXR, bool TAPS>
__device__ __forceinline__ void down_feature(const DNArgs &a, const int8_t *dq,
                                             const uint16_t *ds, uint32_t width, int m,
                                             int row0, int nrows) {
  const int lane = threadIdx.x & 31;
  const uint32_t nb = width / 32, nbmax = a.fmax / 32;
  const int8_t *row = dq + (size_t)m * row_bytes(FMT, width);
  const uint16_t *srow = ds + (size_t)m * nb;
  const int jt = tap_index<TAPS>((uint32_t)m, a.d);
  for (int r0 = 0; r0 < nrows; r0 += MAXR) {
    const int nr = min(MAXR, nrows - r0);
    float acc[MAXR];
#pragma unroll
    for (int r = 0; r < MAXR; ++r) acc[r] = 0.0f;
#pragma unroll 2
    for (uint32_t b = lane; b < nb; b += 32) {
      WBlock<FMT> wd;
      wd.load(row, b);
      const float sw = half_bits_to_float(srow[b]);
#pragma unroll
      for (int r = 0; r < MAXR; ++r) {
        if (r < nr) {
          const size_t slot = (size_t)(row0 + r0 + r);
          const W8 x = ld_cached32(a.hq + slot * a.fmax + 32 * b);
          const float hsc = a.hs[slot * nbmax + b];
          const int is = wd.dot(x);
          acc[r] = __fmaf_rn((float)is, sw * hsc, acc[r]);
          if (TAPS && jt >= 0) a.tap[(slot * kNTap + jt) * nbmax + b] = is;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < MAXR; ++r) {
      const float v = warp_sum(acc[r]);
      if (lane == 0 && r < nr) a.o[(size_t)(row0 + r0 + r) * a.d + m] = v;
    }
  }
}

template <int FMT, int MAXR, bool TAPS>
__global__ void __launch_bounds__(kWarpsPerCta * 32, MAXR <= 2 ? 3 : 2) k_down(const DNArgs a) {
  PlanView P(const_cast<int *>(a.plan), a.E);
  const int total = P.hdr[2];
  const int nwarps = gridDim.x * kWarpsPerCta;
  for (int item = blockIdx.x * kWarpsPerCta + threadIdx.x / 32; item < total; item += nwarps) {
    const int u = item / (int)a.d;
    const int m = item - u * (int)a.d;
    const int e = P.act_e[u];
    const int row0 = P.act_row0[u], nrows = P.act_rows[u];
    if ((uint32_t)e == a.E) {
      down_feature<MOE_FMT_Q8_0, MAXR, TAPS>(a, a.sdq, a.sds, a.fs, m, row0, nrows);
    } else {
      const size_t qoff = (size_t)e * a.d * row_bytes(FMT, a.f);
      const size_t soff = (size_t)e * a.d * (a.f / 32);
      down_feature<FMT, MAXR, TAPS>(a, a.dq + qoff, a.ds + soff, a.f, m, row0, nrows);
    }
  }
}

// y[t][m] = o_shared[t][m] + sum_j w[t,j] * o[pos[t,j]][m], in that order
__global__ void __launch_bounds__(256)
    k_combine(const float *__restrict__ o, const float *__restrict__ w,
              const int32_t *__restrict__ pos, uint32_t T, uint32_t k, uint32_t d, uint32_t R,
              bool shared, const int *__restrict__ plan, float *__restrict__ y) {
  const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (uint64_t)T * d) return;
  if (plan[4] != 1) {  // rejected routing arrays: no expert ran, pos[] is not trusted
    y[i] = 0.0f;
    return;
  }
  const uint32_t t = (uint32_t)(i / d), m = (uint32_t)(i % d);
  float acc = shared ? o[((size_t)R + t) * d + m] : 0.0f;
  for (uint32_t j = 0; j < k; ++j) {
    const int p = pos[(size_t)t * k + j];
    acc = __fmaf_rn(w[(size_t)t * k + j], o[(size_t)p * d + m], acc);
  }
  y[i] = acc;
}

template <typename K>
int persistent_grid(K kernel, int sm_count) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kWarpsPerCta * 32, 0) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return per_sm * sm_count;
}

template <int FMT, int MAXR, bool TAPS>
cudaError_t run_gateup(const Ctx &c, const GUArgs &a) {
  auto kern = k_gateup<FMT, MAXR, TAPS>;
  kern<<<persistent_grid(kern, c.sm_count), kWarpsPerCta * 32, 0, c.stream>>>(a);
  return cudaGetLastError();
}

template <int FMT, int MAXR, bool TAPS>
cudaError_t run_down(const Ctx &c, const DNArgs &a) {
  auto kern = k_down<FMT, MAXR, TAPS>;
  kern<<<persistent_grid(kern, c.sm_count), kWarpsPerCta * 32, 0, c.stream>>>(a);
  return cudaGetLastError();
}

// rows per pass: an expert has at most T rows, and at most kTcMinRows when the
// tensor-core path takes the larger experts
int maxr_for(uint32_t T, bool tc) {
  if (tc && T > kTcMinRows) T = kTcMinRows;
  return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : T <= 8 ? 8 : 16;
}

template <int FMT, int MAXR>
cudaError_t gu_taps(const Ctx &c, const GUArgs &a, bool taps) {
  return taps ? run_gateup<FMT, MAXR, true>(c, a) : run_gateup<FMT, MAXR, false>(c, a);
}
template <int FMT, int MAXR>
cudaError_t dn_taps(const Ctx &c, const DNArgs &a, bool taps) {
  return taps ? run_down<FMT, MAXR, true>(c, a) : run_down<FMT, MAXR, false>(c, a);
}

template <int FMT>
cudaError_t gu_maxr(const Ctx &c, const GUArgs &a, bool taps) {
  switch (maxr_for(c.T, c.L.xperm != 0 && tc_supported(c.desc))) {
    case 1: return gu_taps<FMT, 1>(c, a, taps);
    case 2: return gu_taps<FMT, 2>(c, a, taps);
    case 4: return gu_taps<FMT, 4>(c, a, taps);
    case 8: return gu_taps<FMT, 8>(c, a, taps);
    default: return gu_taps<FMT, 16>(c, a, taps);
  }
}
template <int FMT>
cudaError_t dn_maxr(const Ctx &c, const DNArgs &a, bool taps) {
  switch (maxr_for(c.T, c.L.xperm != 0 && tc_supported(c.desc))) {
    case 1: return dn_taps<FMT, 1>(c, a, taps);
    case 2: return dn_taps<FMT, 2>(c, a, taps);
    case 4: return dn_taps<FMT, 4>(c, a, taps);
    case 8: return dn_taps<FMT, 8>(c, a, taps);
    default: return dn_taps<FMT, 16>(c, a, taps);
  }
}

}  // namespace

cudaError_t launch_gateup(const Ctx &c, const int32_t *perm) {
  if (c.T == 0) return cudaSuccess;
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
  a.xq = (const int8_t *)(c.ws + c.L.xq);
  a.xs = (const float *)(c.ws + c.L.xs);
  a.perm = perm;
  a.h = (float *)(c.ws + c.L.h);
  a.tap = (int32_t *)(c.ws + c.L.tap_gu);
  a.routed_fmt = c.desc.routed_fmt;
  const bool taps = (c.desc.flags & MOE_FLAG_DEBUG_TAPS) != 0;
  return c.desc.routed_fmt == MOE_FMT_Q2S ? gu_maxr<MOE_FMT_Q2S>(c, a, taps)
                                          : gu_maxr<MOE_FMT_Q8_0>(c, a, taps);
}

cudaError_t launch_requant_h(const Ctx &c) {
  const uint32_t slots = c.R + (c.desc.f_shared ? c.T : 0);
  const uint64_t warps = (uint64_t)slots * (c.fmax / 32);
  if (warps == 0) return cudaSuccess;
  k_requant<<<(unsigned)((warps + 7) / 8), 256, 0, c.stream>>>(
      (const float *)(c.ws + c.L.h), slots, c.R, c.desc.f, c.desc.f_shared, c.fmax,
      (int8_t *)(c.ws + c.L.hq), (float *)(c.ws + c.L.hs));
  return cudaGetLastError();
}

cudaError_t launch_down(const Ctx &c) {
  if (c.T == 0) return cudaSuccess;
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
  a.sdq = (const int8_t *)c.wts.s_down.q;
  a.sds = c.wts.s_down.scale;
  a.hq = (const int8_t *)(c.ws + c.L.hq);
  a.hs = (const float *)(c.ws + c.L.hs);
  a.o = (float *)(c.ws + c.L.o);
  a.tap = (int32_t *)(c.ws + c.L.tap_dn);
  const bool taps = (c.desc.flags & MOE_FLAG_DEBUG_TAPS) != 0;
  return c.desc.routed_fmt == MOE_FMT_Q2S ? dn_maxr<MOE_FMT_Q2S>(c, a, taps)
                                          : dn_maxr<MOE_FMT_Q8_0>(c, a, taps);
}

cudaError_t launch_combine(const Ctx &c, const float *w, const int32_t *pos, float *y) {
  const uint64_t n = (uint64_t)c.T * c.desc.d;
  if (n == 0) return cudaSuccess;
  k_combine<<<(unsigned)((n + 255) / 256), 256, 0, c.stream>>>(
      (const float *)(c.ws + c.L.o), w, pos, c.T, c.desc.top_k, c.desc.d, c.R,
      c.desc.f_shared > 0, (const int *)(c.ws + c.L.plan), y);
  return cudaGetLastError();
}

}  // namespace moe
