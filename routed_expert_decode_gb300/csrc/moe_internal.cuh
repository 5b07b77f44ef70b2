// moe_internal.cuh -- device helpers and kernel launchers shared by the
// library's translation units.  Nothing here is shared with the CPU oracle.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int kWarp = 32;
constexpr int kBlock = 32;   // quantisation block (weights and activations)
constexpr int kNTap = 8;     // tapped features per slot when MOE_FLAG_DEBUG_TAPS
constexpr int kSmCount = 152;

// device error word bits
constexpr uint32_t kErrBadIndex = 1u;   // expert index outside [0, E)
constexpr uint32_t kErrBadOffsets = 2u; // off[] not a valid prefix of R rows
constexpr uint32_t kErrTimeout = 4u;    // a bounded wait gave up
constexpr uint32_t kErrBadSlot = 8u;    // a selected expert's weight slot outside [0, n_slots)

// the weight slot of routed expert e (moe_weights.expert_slot; identity without one)
__device__ __forceinline__ int weight_slot(const int32_t *eslot, int e) {
  return eslot ? __ldg(eslot + e) : e;
}

// ---------------------------------------------------------------- plan layout
// int32 array in the workspace describing the active experts of one call.
//   [0] U (experts on the dp4a path, incl. the shared one if there)
//   [1] gate/up work items  [2] down work items  [3] largest routed row count
//   [4] 1 once the routing arrays were validated
//   [5] experts on the tensor-core path  [6] their gate/up tiles  [7] down tiles
//   act_e / act_row0 / act_rows [E+1]: dp4a experts (id E = shared), first slot, rows
//   item_gu[E+2]: exclusive prefix of dp4a gate/up items (features)
//   tc_e / tc_row0 / tc_rows [E+1]: tensor-core experts
//   tc_tile_gu / tc_tile_dn [E+2]: exclusive prefix of their 128x64 tiles
struct PlanView {
  int *hdr, *act_e, *act_row0, *act_rows, *item_gu;
  int *tc_e, *tc_row0, *tc_rows, *tc_tile_gu, *tc_tile_dn;
  __host__ __device__ PlanView(int *base, uint32_t E) {
    hdr = base;
    act_e = base + 8;
    act_row0 = act_e + (E + 1);
    act_rows = act_row0 + (E + 1);
    item_gu = act_rows + (E + 1);
    tc_e = item_gu + (E + 2);
    tc_row0 = tc_e + (E + 1);
    tc_rows = tc_row0 + (E + 1);
    tc_tile_gu = tc_rows + (E + 1);
    tc_tile_dn = tc_tile_gu + (E + 2);
  }
  __host__ __device__ static size_t ints(uint32_t E) { return 8 + 9 * (size_t)(E + 2); }
};

// index u of the dp4a expert whose items [prefix[u], prefix[u+1]) hold `item`
__device__ __forceinline__ int find_slot(const int *prefix, int U, int item) {
  int lo = 0, hi = U;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid;
  }
  return lo;
}

// The plan's dp4a expert list (act_e, act_row0, act_rows, item_gu: 4(E+1)+1
// consecutive ints) copied into shared memory, so that the per-item lookups
// cost no global round trips.
struct SmemPlan {
  const int *e, *row0, *rows, *item;
  __device__ SmemPlan(int *sm, const PlanView &P, uint32_t E) {
    const int n = 4 * (int)(E + 1) + 1;
    for (int i = threadIdx.x; i < n; i += blockDim.x) sm[i] = P.act_e[i];
    __syncthreads();
    e = sm;
    row0 = sm + (E + 1);
    rows = row0 + (E + 1);
    item = rows + (E + 1);
  }
};
inline size_t smem_plan_bytes(uint32_t E) { return sizeof(int) * (4 * (size_t)(E + 1) + 1); }

// Work queues of the persistent expert kernels: pairs of words (items taken,
// CTAs done) in the workspace's fixed sync area (moe.h), zero between calls
// (the last CTA out of a kernel zeroes its pair), clear of the fused decode
// kernel's counters (words [0, 4 + E + 1) and the last two).
constexpr uint32_t kQueueStreamGateup = 2048, kQueueStreamDown = 2050;
constexpr uint32_t kQueueTcGateup = 2052, kQueueTcDown = 2054;
static_assert(4 + 1024 + 1 <= kQueueStreamGateup && kQueueTcDown + 2 <= MOE_SYNC_BYTES / 4 - 2,
              "work queues overlap the fused kernel's counters");

// rows per expert above which an expert runs on the tensor-core path.  Timed on
// the 256-expert layers: 6 for int8 and 2-bit weights (experts of 5-6 rows are
// as fast or faster on the dp4a GEMV, whose weight stream they then join), 4
// for e2m1 (whose GEMV spends more instructions a weight decoding codes)
__host__ __device__ constexpr uint32_t tc_min_rows_for(int32_t routed_fmt) {
  return routed_fmt == MOE_FMT_E2M1 ? 4u : 6u;
}
// calls with fewer tokens run every expert on the dp4a GEMV (no tensor kernel,
// no activation copies launched): measured on the 256-expert layer, the GEMV
// alone was as fast or faster up to 16 tokens a call, the tensor path faster
// from 32
constexpr uint32_t kTcMinTokens = 32;
constexpr uint32_t kTcTileM = 128, kTcTileN = 64;

// ---------------------------------------------------------------- spec-exp
// e^x, bit-reproducible on any IEEE fp32 machine: clamp to [-86, 88];
// n = rint(x * log2e); Cody-Waite reduction r = (x - n*C1) - n*C2 with
// C1 = 355/512 and C2 = fp32(ln2 - C1); degree-7 Taylor polynomial of e^r with
// fp32(1/k!) coefficients by Horner (fma); scaled by an exactly built 2^n.
__device__ __forceinline__ float spec_exp(float x) {
  x = fminf(fmaxf(x, -86.0f), 88.0f);
  const float n = rintf(__fmul_rn(x, 0x1.715476p+0f));
  float r = __fmaf_rn(-n, 0x1.63p-1f, x);
  r = __fmaf_rn(-n, -0x1.bd0106p-13f, r);
  float p = 0x1.a01a02p-13f;            // 1/7!
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f); // 1/6!
  p = __fmaf_rn(p, r, 0x1.111112p-7f);  // 1/5!
  p = __fmaf_rn(p, r, 0x1.555556p-5f);  // 1/4!
  p = __fmaf_rn(p, r, 0x1.555556p-3f);  // 1/3!
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const int ni = __float2int_rn(n);
  return __fmul_rn(p, __int_as_float((ni + 127) << 23));
}

__device__ __forceinline__ float sigmoid_rn(float x) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, spec_exp(-x)));
}

// log(1+y), 0 <= y <= 1: z = y/(2+y), 2z * (1 + z^2/3 + ... + z^14/15) with
// fp32(1/(2n+1)) by Horner (fma) -- bit-reproducible like spec_exp
__device__ __forceinline__ float spec_log1p(float y) {
  const float z = __fdiv_rn(y, __fadd_rn(2.0f, y));
  const float z2 = __fmul_rn(z, z);
  float p = 0x1.111112p-4f;          // 1/15
  p = __fmaf_rn(p, z2, 0x1.3b13b2p-4f);  // 1/13
  p = __fmaf_rn(p, z2, 0x1.745d18p-4f);  // 1/11
  p = __fmaf_rn(p, z2, 0x1.c71c72p-4f);  // 1/9
  p = __fmaf_rn(p, z2, 0x1.24924ap-3f);  // 1/7
  p = __fmaf_rn(p, z2, 0x1.99999ap-3f);  // 1/5
  p = __fmaf_rn(p, z2, 0x1.555556p-2f);  // 1/3
  p = __fmaf_rn(p, z2, 1.0f);
  return __fmul_rn(__fmul_rn(2.0f, z), p);
}

// sqrt(softplus(l)), softplus(l) = max(l, 0) + log1p(e^-|l|)
__device__ __forceinline__ float sqrt_softplus_rn(float l) {
  const float m = l > 0.0f ? l : 0.0f;
  return __fsqrt_rn(__fadd_rn(m, spec_log1p(spec_exp(-fabsf(l)))));
}

// the expert score p of a logit under moe_score `fn`
__device__ __forceinline__ float score_rn(float l, uint32_t fn) {
  return fn == MOE_SCORE_SQRT_SOFTPLUS ? sqrt_softplus_rn(l) : sigmoid_rn(l);
}

// Router logits order (moe_router_logits): the d inputs form segments of
// kRouterSeg; the partial sum of segment g is an fma chain per lane l over
// i = kRouterSeg*g + l + 32j, j ascending (i < d), followed by the lanes'
// pairwise sums over xor distances 16, 8, 4, 2, 1; a logit is the segment sums
// added in ascending g.  router_seg_sums gives every lane of the warp the sums
// of segment g for NT tokens (x rows xr[t]) against one router row, issuing
// the loads of JB consecutive j at a time (the chain order does not change).
constexpr int kRouterSeg = 1024;

template <int NT, int JB>
__device__ __forceinline__ void router_seg_sums(const float *const (&xr)[NT], const float *wrow,
                                                uint32_t g, uint32_t d, int lane, float (&p)[NT]) {
  static_assert(32 % JB == 0, "JB divides the 32 steps of a lane");
  const uint32_t i0 = g * kRouterSeg + (uint32_t)lane;
#pragma unroll
  for (int t = 0; t < NT; ++t) p[t] = 0.0f;
#pragma unroll
  for (int j0 = 0; j0 < 32; j0 += JB) {
    float wv[JB], xv[NT][JB];
#pragma unroll
    for (int j = 0; j < JB; ++j) {
      const uint32_t i = i0 + 32u * (uint32_t)(j0 + j);
      const bool ok = i < d;
      wv[j] = ok ? __ldg(wrow + i) : 0.0f;
#pragma unroll
      for (int t = 0; t < NT; ++t) xv[t][j] = ok ? __ldg(xr[t] + i) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < JB; ++j)
      if (i0 + 32u * (uint32_t)(j0 + j) < d) {
#pragma unroll
        for (int t = 0; t < NT; ++t) p[t] = __fmaf_rn(xv[t][j], wv[j], p[t]);
      }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int t = 0; t < NT; ++t) p[t] = __fadd_rn(p[t], __shfl_xor_sync(0xffffffffu, p[t], o));
  }
}

// one 32-element block: scale = amax/127, q = clamp(round_half_away(x/scale))
__device__ __forceinline__ int quant_one(float x, float scale) {
  if (scale == 0.0f) return 0;
  float v = roundf(__fdiv_rn(x, scale));
  v = fminf(fmaxf(v, -127.0f), 127.0f);
  return (int)v;
}

__device__ __forceinline__ float half_bits_to_float(uint16_t b) {
  return __half2float(__ushort_as_half(b));
}

// ---------------------------------------------------------------- loads
struct W8 {
  uint32_t v[8];
};

// 32 bytes, read-only, streamed (no L1 allocation)
__device__ __forceinline__ W8 ld_stream32(const void *p) {
  W8 w;
  asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(w.v[0]), "=r"(w.v[1]), "=r"(w.v[2]), "=r"(w.v[3]), "=r"(w.v[4]), "=r"(w.v[5]),
        "=r"(w.v[6]), "=r"(w.v[7])
      : "l"(p));
  return w;
}

// 32 bytes, read-only, cached (activations reused by many warps)
__device__ __forceinline__ W8 ld_cached32(const void *p) {
  W8 w;
  asm("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(w.v[0]), "=r"(w.v[1]), "=r"(w.v[2]), "=r"(w.v[3]), "=r"(w.v[4]), "=r"(w.v[5]),
        "=r"(w.v[6]), "=r"(w.v[7])
      : "l"(p));
  return w;
}

// as ld_cached32, but issued exactly where written (volatile): keeps the
// compiler from hoisting a whole unrolled loop's activation loads ahead of use
__device__ __forceinline__ W8 ld_cached32_here(const void *p) {
  W8 w;
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w.v[0]), "=r"(w.v[1]), "=r"(w.v[2]), "=r"(w.v[3]), "=r"(w.v[4]),
                 "=r"(w.v[5]), "=r"(w.v[6]), "=r"(w.v[7])
               : "l"(p));
  return w;
}

__device__ __forceinline__ uint2 ld_stream8(const void *p) {
  uint2 w;
  asm("ld.global.nc.L1::no_allocate.v2.b32 {%0,%1}, [%2];" : "=r"(w.x), "=r"(w.y) : "l"(p));
  return w;
}

// ---------------------------------------------------------------- block dots
// Weight block in registers, per format.  Q8_0: 8 words of int8.  Q2S: the
// 8 code bytes spread to 8 words of one code (0..3) per byte lane.
template <int FMT>
struct WBlock;

template <>
struct WBlock<MOE_FMT_Q8_0> {
  W8 w;
  static constexpr int kRowBytesPer32 = 32;
  static constexpr bool kNeedSum = false;
  __device__ __forceinline__ void load(const int8_t *row, int b) { w = ld_stream32(row + 32 * b); }
  __device__ __forceinline__ void prep() {}
  __device__ __forceinline__ int dot(const W8 &x, int /*sum_x*/) const {
    int s = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) s = __dp4a((int)w.v[q], (int)x.v[q], s);
    return s;
  }
};

template <>
struct WBlock<MOE_FMT_Q2S> {
  uint2 c;
  uint32_t t[8];
  static constexpr int kRowBytesPer32 = 8;
  static constexpr bool kNeedSum = true;
  __device__ __forceinline__ void load(const int8_t *row, int b) { c = ld_stream8(row + 8 * b); }
  // Byte j of code word g (codes 16g .. 16g+15, LSB first) holds codes
  // 16g+4j .. 16g+4j+3; t[4g+i] = (word >> 2i) & 0x03030303 has code 16g+4j+i
  // in byte j, which lines up with activations stored 16-code-group transposed
  // (byte 4i+j of a group = code 4j+i).  Done once per block, reused by every row.
  __device__ __forceinline__ void prep() {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      t[i] = (c.x >> (2 * i)) & 0x03030303u;
      t[4 + i] = (c.y >> (2 * i)) & 0x03030303u;
    }
  }
  // sum_i (2c_i - 3) x_i = 2 sum c_i x_i - 3 sum x_i, exact in int32; x in the
  // transposed order
  __device__ __forceinline__ int dot(const W8 &xt, int sum_x) const {
    int sc = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) sc = __dp4a((int)t[q], (int)xt.v[q], sc);
    return 2 * sc - 3 * sum_x;
  }
};

// prmt.b32 in its generic mode: byte n of the result is byte (c >> 4n) & 7 of
// {b, a} -- or, when bit 4n+3 of c is set, that byte's sign bit replicated
// (the CUDA intrinsic __byte_perm ignores that bit)
__device__ __forceinline__ uint32_t prmt_sx(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Four 4-bit e2m1 codes (the low 16 bits of w, code j at bits 4j..4j+3: sign
// bit 3, exponent bits 1-2 with bias 1, mantissa bit 0) -> four bytes holding
// TWICE the value plus 12: 2v is one of 0, 1, 2, 3, 4, 6, 8, 12 or its
// negative, so every byte is 0..24.  One byte permute looks up the positive
// and one the negative table (indexed by the code's low 3 bits); a third, with
// the sign bit as its sign-replicate flag over bytes 0x80, gives 0xFF for a
// negative code and 0x80 for a positive one, and since both tables' bytes are
// below 128 that word selects between them bit by bit.
__device__ __forceinline__ uint32_t e2m1x4_biased(uint32_t w) {
  const uint32_t sel = w & 0x7777u;
  const uint32_t pos = __byte_perm(0x0F0E0D0Cu, 0x18141210u, sel);  // 12 + (0,1,2,3,4,6,8,12)
  const uint32_t neg = __byte_perm(0x090A0B0Cu, 0x00040608u, sel);  // 12 - (0,1,2,3,4,6,8,12)
  const uint32_t m = prmt_sx(0x80808080u, 0x80808080u, w & 0xFFFFu);
  return (m & neg) | (~m & pos);
}

// e2m1: 16 bytes = 32 codes (low nibble first); prep() decodes them once per
// block into 8 words of biased bytes 2v + 12 (natural order, like the int8
// activation codes), and dot = sum (2v + 12) x - 12 sum x = sum 2v x, exact.
// The block dot is of twice the weights: kScaleMul halves the weight scale.
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  uint4 w;
  asm("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
      : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
      : "l"(p));
  return w;
}

template <>
struct WBlock<MOE_FMT_E2M1> {
  uint4 c;
  uint32_t t[8];
  static constexpr int kRowBytesPer32 = 16;
  static constexpr bool kNeedSum = true;
  __device__ __forceinline__ void load(const int8_t *row, int b) { c = ld_stream16(row + 16 * b); }
  __device__ __forceinline__ void prep() {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      t[2 * q] = e2m1x4_biased(w[q]);
      t[2 * q + 1] = e2m1x4_biased(w[q] >> 16);
    }
  }
  __device__ __forceinline__ int dot(const W8 &x, int sum_x) const {
    int s = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) s = __dp4a((int)t[q], (int)x.v[q], s);
    return s - 12 * sum_x;
  }
};

// weight-scale factor of a format's block dots (e2m1 dots are of twice the values)
template <int FMT>
__host__ __device__ constexpr float scale_mul() { return FMT == MOE_FMT_E2M1 ? 0.5f : 1.0f; }

// sum of the 32 int8 codes of an activation block
__device__ __forceinline__ int block_sum(const W8 &x) {
  int s = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) s = __dp4a(0x01010101, (int)x.v[q], s);
  return s;
}

__host__ __device__ inline size_t row_bytes(int fmt, uint32_t K) {
  return fmt == MOE_FMT_Q2S ? K / 4 : fmt == MOE_FMT_E2M1 ? K / 2 : K;
}

// tapped feature j of a row of `width` outputs
__host__ __device__ inline uint32_t tap_feature(uint32_t j, uint32_t width) {
  return (uint32_t)(((uint64_t)j * width / kNTap + j) % width);
}

// ---------------------------------------------------------------- dependent launch
// The multi-kernel path is a chain of kernels on one stream.  Each kernel after
// the first is launched with programmatic stream serialization: it may start
// (and be scheduled onto free SM resources) once every CTA of its predecessor
// has started and triggered, so its launch overlaps the predecessor's tail.
// Every such kernel calls pdl_wait() -- which returns once the predecessor grid
// has completed and its writes are visible -- before reading what the chain
// produced, and in any case before it exits, so each kernel's completion
// still implies its predecessors' (the dependency stays transitive).
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// launch `kern` on `stream`, as a programmatic dependent of the stream's
// previous kernel when `dep`
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, bool dep, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = dep ? attr : nullptr;
  cfg.numAttrs = dep ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- launchers
struct Ctx {
  moe_desc desc;
  moe_weights wts;
  uint32_t T, R;
  uint32_t fmax;
  uint32_t wexp;  // expert-sized slots in the routed weight planes (E without a slot table)
  uint8_t *ws;
  moe_ws_layout L;
  cudaStream_t stream;
  int sm_count;
  // routed experts this call computes, [e_lo, e_hi), and whether it adds the
  // shared expert (an expert-parallel rank's share; [0, E) and true otherwise)
  uint32_t e_lo, e_hi;
  bool shared_on;
  // a kernel of this call is already on the stream: the next one is launched as
  // its programmatic dependent (launch_k)
  mutable bool chained;
};

cudaError_t launch_route(const Ctx &c, const float *logits, const float *bias, int32_t *idx,
                         float *w);
cudaError_t launch_router_logits(const moe_desc &d, const float *w_router, const float *x,
                                 uint32_t T, float *logits, cudaStream_t stream);
cudaError_t launch_permute(const Ctx &c, const int32_t *idx, int32_t *off, int32_t *perm,
                           int32_t *pos, uint32_t *err);
cudaError_t launch_plan(const Ctx &c, const int32_t *off, const int32_t *idx,
                        const int32_t *perm, const int32_t *pos, uint32_t *err);
// tensor-core path (expert_tc.cu)
bool tc_supported(const moe_desc &D);
// the weight planes the tensor maps read are 16-byte aligned (else no expert of
// the call takes the tensor path)
bool tc_weights_aligned(const Ctx &c);
bool tc_possible(const moe_desc &D, uint32_t T);
cudaError_t launch_tc_prepare(const Ctx &c, const int32_t *perm);
cudaError_t launch_tc(const Ctx &c, int mat);
cudaError_t launch_quant_x(const Ctx &c, const float *x);
cudaError_t launch_gateup(const Ctx &c, const int32_t *perm);
// the streamed GEMV (weights through shared memory by bulk copies): eligible
// calls, and its gate/up and down launches
bool stream_gateup_ok(const Ctx &c);
bool stream_down_ok(const Ctx &c);
cudaError_t launch_gateup_stream(const Ctx &c, const int32_t *perm);
cudaError_t launch_down_stream(const Ctx &c);
cudaError_t launch_requant_h(const Ctx &c);
cudaError_t launch_down(const Ctx &c);
cudaError_t launch_combine(const Ctx &c, const float *w, const int32_t *pos,
                           const int32_t *idx, float *y);

// fused single-kernel decode (T <= 2): decode_fused.cu
size_t fused_sync_ints(const moe_desc *d);
bool fused_eligible(const Ctx &c);
// w_router non-null: the kernel computes the router logits itself from x and
// stores them to logits_out (`logits` is unused); else `logits` is the input
cudaError_t launch_decode_fused(const Ctx &c, const float *x, const float *logits,
                                const float *bias, float *y, const float *w_router,
                                float *logits_out);

moe_status layer_on_workspace(const moe_desc *desc, const moe_weights *wts, const float *x,
                              const float *logits, const float *bias, uint32_t T, float *y,
                              void *ws, size_t ws_bytes, void *stream);
void set_last_error(const char *msg);
// moe_layer_noalloc's static scratch on the current device, or null when no such
// call has set it up there (moe_noalloc.cu); never touches CUDA before that
void *noalloc_scratch_current();

// expert cache internals for moe_stream_layer (expert_cache.cu)
bool cache_layer_routed(const moe_cache *c, uint32_t layer, moe_weights *w);
const moe_desc *cache_desc(const moe_cache *c);
int32_t *cache_pinned(moe_cache *c, size_t n);

}  // namespace moe
