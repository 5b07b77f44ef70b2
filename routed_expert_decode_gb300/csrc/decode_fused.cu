// decode_fused.cu -- the whole layer for one or two tokens in one persistent kernel.
//
// Single-token decode moves ~361 MB of expert weights (8 routed experts + the
// shared expert of a GLM-5.2-sized layer) and almost no arithmetic, so the
// layer is bound by HBM bandwidth and by anything that leaves HBM idle:
// launch gaps between small kernels, the router's latency, and the drain/ramp
// between the gate/up and the down projection.  This kernel removes all three.
//
//  * One CTA per SM (cooperative launch, all CTAs co-resident), 8 consumer warps
//    and 1 producer warp.  The producer lane streams weight rows with
//    cp.async.bulk (the bulk-copy/TMA engine, one-CTA copies, no multicast) into
//    a ring of shared-memory stages guarded by mbarriers; consumers compute from
//    shared memory with dp4a.
//  * Work comes from one global queue, handed out in this order: gate/up items
//    of the shared expert (they need no routing), gate/up items of the routed
//    experts, then down items of every expert.  A gate/up item is 32 features
//    of one expert (one int8 block of h, requantised by the CTA that computed
//    it); a down item is a chunk of output rows of one expert.
//  * CTA 0's consumer warps route the tokens first (sigmoid + bias, top-k,
//    stable permutation) and publish the active-expert list with a release
//    flag; meanwhile every other CTA is already streaming the shared expert.
//  * A down item needs its expert's h complete: consumers wait on a per-expert
//    counter, while the producer keeps prefetching weights (which do not depend
//    on h).  Because every gate/up item is handed out before any down item and
//    all CTAs are resident, every such wait ends.
//  * The combine (y = o_shared + sum_j w_j o_j, fixed order) of an output chunk
//    is done by the CTA that lands the chunk's last contribution.
//  * Every wait is bounded; on timeout the kernel flags kErrTimeout and exits.
// Per-expert batches of the selected experts only, read once per call: the
// indexed per-expert FFN of NeutronStar README, "MTP speculative decoding".
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxT = 2;
constexpr int kBFeat = 8;        // features per gate/up stage: one per consumer warp
constexpr int kBItemFeat = 32;   // features per gate/up item: one quantisation block
constexpr int kMaxStages = 4;
constexpr int kSpinIters = 1 << 26;                // iteration cap of every wait
constexpr long long kWaitCycles = 4000000000ll;     // ~2 s at 2 GHz: a wait gives up after this
constexpr long long kStallTestCycles = 20000000ll;  // ~10 ms under MOE_FLAG_TEST_STALL

enum : int { kKindB = 0, kKindC = 1, kKindEnd = 2 };

struct StageDesc {
  int kind;
  int e;           // expert id, E = shared expert
  int first;       // B: first feature of the stage; C: first output row
  int count;       // B: features (8); C: output rows
  int sub;         // B: sub-stage in the item (0..3)
  int item_first;  // B: first feature of the item; C: chunk index
  int nrows;       // token rows of this expert
  int n_contrib;   // C: experts contributing to each chunk
  int slot[kMaxT];
  int tok[kMaxT];
};

struct FusedArgs {
  uint32_t E, k, d, f, fs, T, R, fmax;
  float s;
  const float *x, *logits, *bias;
  const int8_t *gq, *uq, *dq, *sgq, *suq, *sdq;
  const uint16_t *gs, *us, *ds, *sgs, *sus, *sds;
  float *y;
  int32_t *idx;
  float *w;
  int32_t *off, *perm, *pos;
  int8_t *xq;
  float *xs;
  int8_t *hq;
  float *hs;
  float *o;
  int *plan;
  uint32_t *sync;  // [0] queue, [1] route flag, [4..4+E] expert ready, then chunk counters
  uint32_t *err;
  uint32_t c_rows, n_chunks, n_stages, stage_bytes;
  long long wait_cycles;  // budget of every bounded wait
  int stall_test;         // MOE_FLAG_TEST_STALL: never publish the routing result
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// bounded wait for completion of the phase with the given parity
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long long budget) {
  const uint32_t a = smem_u32(bar);
  const long long t0 = clock64();
  for (int i = 0; i < kSpinIters; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
    if (clock64() - t0 > budget) return false;
  }
  return false;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// bounded wait until *p >= target (acquire); false on timeout
__device__ __forceinline__ bool wait_geq(const uint32_t *p, uint32_t target, long long budget) {
  const long long t0 = clock64();
  for (int i = 0; i < kSpinIters; ++i) {
    if (ld_acquire(p) >= target) return true;
    if (clock64() - t0 > budget) return false;
    __nanosleep(64);
  }
  return false;
}

__device__ __forceinline__ int ld_cg_i32(const int *p) { return __ldcg(p); }

// a bounded wait gave up: flag the error word (kErrTimeout plus the wait site in
// bits 8..15) and keep the first site / CTA / detail in sync[2], sync[3]
__device__ __noinline__ void report_timeout(const FusedArgs &a, uint32_t site, uint32_t detail) {
  atomicOr(a.err, kErrTimeout | (1u << (8 + site)));
  if (atomicCAS(&a.sync[2], 0u, (site << 24) | (blockIdx.x & 0xFFFFFFu)) == 0u)
    a.sync[3] = detail;
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

__device__ __forceinline__ W8 lds32(const int8_t *p) {
  const uint4 a = *reinterpret_cast<const uint4 *>(p);
  const uint4 b = *reinterpret_cast<const uint4 *>(p + 16);
  W8 w;
  w.v[0] = a.x; w.v[1] = a.y; w.v[2] = a.z; w.v[3] = a.w;
  w.v[4] = b.x; w.v[5] = b.y; w.v[6] = b.z; w.v[7] = b.w;
  return w;
}

__device__ __forceinline__ int dot8(const W8 &a, const W8 &b) {
  int s = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) s = __dp4a((int)a.v[q], (int)b.v[q], s);
  return s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------- routing (CTA 0)
// Warp t routes token t; then the consumer threads build the stable permutation
// (R <= 64 rows: rank by comparison), off[], and the active-expert list.
__device__ void route_tokens(const FusedArgs &a, int *s_idx, float *s_w) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t E = a.E, k = a.k;
  if (warp < (int)a.T) {
    const int t = warp;
    const float *l = a.logits + (size_t)t * E;
    const int nper = (int)((E + 31) / 32);
    float lv[32], bv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {  // issue every load before any use
      const uint32_t e = (uint32_t)lane + 32u * i;
      const bool ok = i < nper && e < E;
      lv[i] = ok ? l[e] : 0.0f;
      bv[i] = ok ? a.bias[e] : 0.0f;
    }
    float c[32], sg[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t e = (uint32_t)lane + 32u * i;
      c[i] = -INFINITY;
      sg[i] = 0.0f;
      if (i < nper && e < E) {
        sg[i] = sigmoid_rn(lv[i]);
        c[i] = __fadd_rn(sg[i], bv[i]);
      }
    }
    uint32_t taken = 0;
    float my_sigma = 0.0f;
    for (uint32_t j = 0; j < k; ++j) {
      float bc = -INFINITY, bs = 0.0f;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (i < nper && !((taken >> i) & 1u) && c[i] > bc) {
          bc = c[i];
          be = lane + 32 * i;
          bs = sg[i];
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float oc = __shfl_xor_sync(0xffffffffu, bc, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        const float os = __shfl_xor_sync(0xffffffffu, bs, o);
        if (oc > bc || (oc == bc && oe < be)) {
          bc = oc;
          be = oe;
          bs = os;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if ((uint32_t)lane == j) my_sigma = bs;
      if (lane == 0) s_idx[t * k + j] = be;
    }
    float sum = 0.0f;
    for (uint32_t j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, my_sigma, j));
    if ((uint32_t)lane < k) s_w[t * k + lane] = __fmul_rn(a.s, __fdiv_rn(my_sigma, sum));
  }
  consumer_sync();
  const int R = (int)a.R;
  PlanView P(a.plan, E);
  // stable rank of each (token, slot) row by expert
  if (tid < R) {
    const int e = s_idx[tid];
    int rank = 0;
    for (int r = 0; r < R; ++r) {
      const int er = s_idx[r];
      rank += (er < e || (er == e && r < tid)) ? 1 : 0;
    }
    a.idx[tid] = e;
    a.w[tid] = s_w[tid];
    a.pos[tid] = rank;
    a.perm[rank] = tid;
  }
  // off[e] = rows routed to experts below e
  for (uint32_t e = tid; e <= E; e += kConsumerWarps * 32) {
    int c = 0;
    for (int r = 0; r < R; ++r) c += s_idx[r] < (int)e ? 1 : 0;
    a.off[e] = c;
  }
  // active list: one entry per distinct expert, ascending
  if (tid < R) {
    const int e = s_idx[tid];
    bool first = true;
    int below = 0, rows = 0;
    for (int r = 0; r < R; ++r) {
      const int er = s_idx[r];
      if (er == e) {
        ++rows;
        if (r < tid) first = false;
      }
    }
    if (first) {
      // distinct experts smaller than e
      for (int r = 0; r < R; ++r) {
        const int er = s_idx[r];
        if (er < e) {
          bool first_r = true;
          for (int q = 0; q < r; ++q)
            if (s_idx[q] == er) first_r = false;
          below += first_r ? 1 : 0;
        }
      }
      int row0 = 0;
      for (int r = 0; r < R; ++r) row0 += s_idx[r] < e ? 1 : 0;
      P.act_e[below] = e;
      P.act_row0[below] = row0;
      P.act_rows[below] = rows;
    }
  }
  if (tid == 0) {
    int U = 0;
    for (int r = 0; r < R; ++r) {
      bool first_r = true;
      for (int q = 0; q < r; ++q)
        if (s_idx[q] == s_idx[r]) first_r = false;
      U += first_r ? 1 : 0;
    }
    P.hdr[0] = U;  // routed experts only
    P.hdr[4] = 1;
  }
  __threadfence();
  consumer_sync();
  if (tid == 0 && !a.stall_test) st_release(&a.sync[1], 1u);
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(kThreads, 1) k_decode_fused(const FusedArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t T = a.T, d = a.d, nb = d / 32, fmax = a.fmax;
  const uint32_t NS = a.n_stages;
  // shared-memory carve-up
  uint8_t *stages = smem;
  int8_t *xq_s = (int8_t *)(stages + (size_t)NS * a.stage_bytes);
  float *xs_s = (float *)(xq_s + (size_t)kMaxT * d);
  int8_t *hq_s = (int8_t *)(xs_s + (size_t)kMaxT * nb);
  float *hs_s = (float *)(hq_s + (size_t)kMaxT * fmax);
  float *h_tile = hs_s + (size_t)kMaxT * (fmax / 32);
  StageDesc *desc = (StageDesc *)(h_tile + kMaxT * kBItemFeat);
  uint64_t *full = (uint64_t *)(desc + kMaxStages);
  uint64_t *empty = full + kMaxStages;
  volatile int *s_misc = (volatile int *)(empty + kMaxStages);  // [0] abort, [1] chunk is last
  int *s_idx = (int *)(s_misc + 4);                             // [R]
  float *s_w = (float *)(s_idx + 64);                           // [R]

  if (tid == 0) {
    for (uint32_t i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    s_misc[0] = 0;
    s_misc[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const uint32_t n_sh = a.fs / kBItemFeat;          // shared-expert gate/up items
  const uint32_t fb = a.f / kBItemFeat;              // gate/up items per routed expert
  PlanView P(a.plan, a.E);

  if (warp == kConsumerWarps) {
    // ============================ producer (one lane)
    if (lane != 0) return;
    uint32_t g = 0;  // stages issued
    bool routed = false;
    uint32_t U = 0, NB = 0, total = 0;
    for (;;) {
      const uint32_t item = atomicAdd(&a.sync[0], 1u);
      if (!routed && item >= n_sh) {
        if (!wait_geq(&a.sync[1], 1u, a.wait_cycles)) {
          report_timeout(a, 1, item);
          s_misc[0] = 1;
        } else {
          U = (uint32_t)ld_cg_i32(&P.hdr[0]);
          NB = n_sh + U * fb;
          total = NB + (U + (a.fs ? 1u : 0u)) * a.n_chunks;
          routed = true;
        }
      }
      const bool end = s_misc[0] || (routed && item >= total);
      StageDesc dsc;
      dsc.kind = kKindEnd;
      int nsub = 1;
      if (!end) {
        // shared-expert gate/up items come first and are known before routing (NB is
        // only known after it), so test them against n_sh before NB
        if (item < n_sh || item < NB) {  // gate/up item
          dsc.kind = kKindB;
          if (item < n_sh) {
            dsc.e = (int)a.E;
            dsc.item_first = (int)(item * kBItemFeat);
            dsc.nrows = (int)T;
            for (uint32_t r = 0; r < T; ++r) {
              dsc.slot[r] = (int)(a.R + r);
              dsc.tok[r] = (int)r;
            }
          } else {
            const uint32_t u = (item - n_sh) / fb;
            dsc.e = ld_cg_i32(&P.act_e[u]);
            dsc.item_first = (int)(((item - n_sh) % fb) * kBItemFeat);
            const int row0 = ld_cg_i32(&P.act_row0[u]);
            dsc.nrows = ld_cg_i32(&P.act_rows[u]);
            for (int r = 0; r < dsc.nrows; ++r) {
              dsc.slot[r] = row0 + r;
              dsc.tok[r] = ld_cg_i32(&a.perm[row0 + r]) / (int)a.k;
            }
          }
          nsub = kBItemFeat / kBFeat;
        } else {  // down item
          const uint32_t c = item - NB;
          uint32_t uc = c / a.n_chunks;
          const uint32_t chunk = c % a.n_chunks;
          dsc.kind = kKindC;
          dsc.item_first = (int)chunk;
          dsc.first = (int)(chunk * a.c_rows);
          dsc.count = (int)min(a.c_rows, d - chunk * a.c_rows);
          dsc.n_contrib = (int)(U + (a.fs ? 1u : 0u));
          if (a.fs && uc == 0) {
            dsc.e = (int)a.E;
            dsc.nrows = (int)T;
            for (uint32_t r = 0; r < T; ++r) {
              dsc.slot[r] = (int)(a.R + r);
              dsc.tok[r] = (int)r;
            }
          } else {
            if (a.fs) uc -= 1;
            dsc.e = ld_cg_i32(&P.act_e[uc]);
            const int row0 = ld_cg_i32(&P.act_row0[uc]);
            dsc.nrows = ld_cg_i32(&P.act_rows[uc]);
            for (int r = 0; r < dsc.nrows; ++r) {
              dsc.slot[r] = row0 + r;
              dsc.tok[r] = ld_cg_i32(&a.perm[row0 + r]) / (int)a.k;
            }
          }
        }
      }
      for (int sub = 0; sub < nsub; ++sub) {
        const uint32_t st = g % NS, use = g / NS;
        if (use > 0 && !mbar_wait(&empty[st], (use - 1) & 1u, a.wait_cycles)) {
          report_timeout(a, 2, g);
          s_misc[0] = 1;
          dsc.kind = kKindEnd;
        }
        dsc.sub = sub;
        uint8_t *buf = stages + (size_t)st * a.stage_bytes;
        if (dsc.kind == kKindB) {
          dsc.first = dsc.item_first + sub * kBFeat;
          dsc.count = kBFeat;
          const bool sh = dsc.e == (int)a.E;
          const size_t row = sh ? (size_t)dsc.first : (size_t)dsc.e * a.f + dsc.first;
          const int8_t *g_src = (sh ? a.sgq : a.gq) + row * d;
          const int8_t *u_src = (sh ? a.suq : a.uq) + row * d;
          const uint16_t *gs_src = (sh ? a.sgs : a.gs) + row * nb;
          const uint16_t *us_src = (sh ? a.sus : a.us) + row * nb;
          const uint32_t qb = kBFeat * d, sb = kBFeat * nb * 2;
          desc[st] = dsc;
          mbar_expect_tx(&full[st], 2 * qb + 2 * sb);
          bulk_g2s(buf, g_src, qb, &full[st]);
          bulk_g2s(buf + qb, u_src, qb, &full[st]);
          bulk_g2s(buf + 2 * qb, gs_src, sb, &full[st]);
          bulk_g2s(buf + 2 * qb + sb, us_src, sb, &full[st]);
        } else if (dsc.kind == kKindC) {
          const bool sh = dsc.e == (int)a.E;
          const uint32_t K = sh ? a.fs : a.f;
          const size_t row = sh ? (size_t)dsc.first : (size_t)dsc.e * d + dsc.first;
          const int8_t *q_src = (sh ? a.sdq : a.dq) + row * K;
          const uint16_t *s_src = (sh ? a.sds : a.ds) + row * (K / 32);
          const uint32_t qb = dsc.count * K, sb = dsc.count * (K / 32) * 2;
          desc[st] = dsc;
          mbar_expect_tx(&full[st], qb + sb);
          bulk_g2s(buf, q_src, qb, &full[st]);
          bulk_g2s(buf + qb, s_src, sb, &full[st]);
        } else {
          desc[st] = dsc;
          mbar_arrive(&full[st]);
        }
        ++g;
      }
      if (dsc.kind == kKindEnd) return;
    }
  }

  // ============================ consumers (warps 0..7)
  if (blockIdx.x == 0) route_tokens(a, s_idx, s_w);
  // quantise x for this CTA (identical in every CTA); CTA 0 also publishes it
  for (uint32_t b = warp; b < T * nb; b += kConsumerWarps) {
    const uint32_t t = b / nb, bb = b % nb;
    const float v = a.x[(size_t)t * d + 32 * bb + lane];
    float amax = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = __fdiv_rn(amax, 127.0f);
    const int8_t q = (int8_t)quant_one(v, sc);
    xq_s[(size_t)t * d + 32 * bb + lane] = q;
    if (lane == 0) xs_s[t * nb + bb] = sc;
    if (blockIdx.x == 0) {
      a.xq[(size_t)t * d + 32 * bb + lane] = q;
      if (lane == 0) a.xs[t * nb + bb] = sc;
    }
  }
  consumer_sync();

  bool route_seen = blockIdx.x == 0;
  uint32_t g = 0;
  for (;; ++g) {
    const uint32_t st = g % NS, use = g / NS;
    if (!mbar_wait(&full[st], use & 1u, a.wait_cycles)) {
      report_timeout(a, 3, g);
      return;
    }
    const StageDesc dsc = desc[st];
    if (dsc.kind == kKindEnd) return;
    const uint8_t *buf = stages + (size_t)st * a.stage_bytes;
    const int nr = dsc.nrows;
    if (dsc.kind == kKindB) {
      // ---- gate/up: warp w owns feature first + w
      const int8_t *gc = (const int8_t *)buf + (size_t)warp * d;
      const int8_t *uc = (const int8_t *)buf + (size_t)kBFeat * d + (size_t)warp * d;
      const uint16_t *gsc = (const uint16_t *)(buf + 2 * kBFeat * d) + (size_t)warp * nb;
      const uint16_t *usc = (const uint16_t *)(buf + 2 * kBFeat * d) + (size_t)kBFeat * nb +
                            (size_t)warp * nb;
      float accg[kMaxT] = {0.0f, 0.0f}, accu[kMaxT] = {0.0f, 0.0f};
      for (uint32_t b = lane; b < nb; b += 32) {
        const W8 wg = lds32(gc + 32 * b), wu = lds32(uc + 32 * b);
        const float sg = half_bits_to_float(gsc[b]), su = half_bits_to_float(usc[b]);
#pragma unroll
        for (int r = 0; r < kMaxT; ++r) {
          if (r < nr) {
            const int t = dsc.tok[r];
            const W8 xv = lds32(xq_s + (size_t)t * d + 32 * b);
            const float xsc = xs_s[t * nb + b];
            accg[r] = __fmaf_rn((float)dot8(wg, xv), sg * xsc, accg[r]);
            accu[r] = __fmaf_rn((float)dot8(wu, xv), su * xsc, accu[r]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kMaxT; ++r) {
        const float gv = warp_sum(accg[r]), uv = warp_sum(accu[r]);
        if (lane == 0 && r < nr)
          h_tile[r * kBItemFeat + (dsc.first - dsc.item_first) + warp] =
              __fmul_rn(__fdiv_rn(gv, __fadd_rn(1.0f, spec_exp(-gv))), uv);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (dsc.sub == kBItemFeat / kBFeat - 1) {
        // the item's 32 features are done: requantise h (one warp per row)
        consumer_sync();
        if (warp < nr) {
          const float v = h_tile[warp * kBItemFeat + lane];
          float amax = fabsf(v);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          const float sc = __fdiv_rn(amax, 127.0f);
          const size_t slot = (size_t)dsc.slot[warp];
          a.hq[slot * fmax + dsc.item_first + lane] = (int8_t)quant_one(v, sc);
          if (lane == 0) a.hs[slot * (fmax / 32) + dsc.item_first / 32] = sc;
          __threadfence();
        }
        consumer_sync();
        if (tid == 0) atomicAdd(&a.sync[4 + dsc.e], 1u);
      }
    } else {
      // ---- down: wait for the expert's h, stage its codes, dot, combine
      const bool sh = dsc.e == (int)a.E;
      const uint32_t K = sh ? a.fs : a.f, kb = K / 32;
      if (tid == 0) {
        if (!wait_geq(&a.sync[4 + dsc.e], K / kBItemFeat, a.wait_cycles)) {
          report_timeout(a, 4, ((uint32_t)dsc.e << 16) | __ldcg(&a.sync[4 + dsc.e]));
          s_misc[0] = 1;
        } else if (!route_seen && !wait_geq(&a.sync[1], 1u, a.wait_cycles)) {
          report_timeout(a, 5, 0);
          s_misc[0] = 1;
        }
      }
      consumer_sync();
      route_seen = true;
      if (s_misc[0]) return;  // the producer sees the flag and ends too
      for (int r = 0; r < nr; ++r) {
        const size_t slot = (size_t)dsc.slot[r];
        const int4 *src = (const int4 *)(a.hq + slot * fmax);
        int4 *dst = (int4 *)(hq_s + (size_t)r * fmax);
        for (uint32_t i = tid; i < K / 16; i += kConsumerWarps * 32) dst[i] = __ldcg(src + i);
        for (uint32_t i = tid; i < kb; i += kConsumerWarps * 32)
          hs_s[r * (fmax / 32) + i] = __ldcg(a.hs + slot * (fmax / 32) + i);
      }
      consumer_sync();
      const int8_t *qc = (const int8_t *)buf;
      const uint16_t *sc = (const uint16_t *)(buf + (size_t)dsc.count * K);
      for (int m = warp; m < dsc.count; m += kConsumerWarps) {
        float acc[kMaxT] = {0.0f, 0.0f};
        for (uint32_t b = lane; b < kb; b += 32) {
          const W8 wd = lds32(qc + (size_t)m * K + 32 * b);
          const float sw = half_bits_to_float(sc[(size_t)m * kb + b]);
#pragma unroll
          for (int r = 0; r < kMaxT; ++r)
            if (r < nr) {
              const W8 hv = lds32(hq_s + (size_t)r * fmax + 32 * b);
              acc[r] = __fmaf_rn((float)dot8(wd, hv), sw * hs_s[r * (fmax / 32) + b], acc[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < kMaxT; ++r) {
          const float v = warp_sum(acc[r]);
          if (lane == 0 && r < nr) a.o[(size_t)dsc.slot[r] * d + dsc.first + m] = v;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      __threadfence();
      consumer_sync();
      if (tid == 0) {
        const uint32_t old = atomicAdd(&a.sync[4 + a.E + 1 + dsc.item_first], 1u);
        const int last = old + 1 == (uint32_t)dsc.n_contrib;
        if (last) __threadfence();
        s_misc[1] = last;
      }
      consumer_sync();
      if (s_misc[1]) {
        // combine this chunk for every token: shared first, then slots in order
        for (uint32_t i = tid; i < T * (uint32_t)dsc.count; i += kConsumerWarps * 32) {
          const uint32_t t = i / dsc.count, m = dsc.first + i % dsc.count;
          float acc = a.fs ? __ldcg(a.o + ((size_t)a.R + t) * d + m) : 0.0f;
          for (uint32_t j = 0; j < a.k; ++j) {
            const int p = __ldcg(a.pos + t * a.k + j);
            acc = __fmaf_rn(__ldcg(a.w + t * a.k + j), __ldcg(a.o + (size_t)p * d + m), acc);
          }
          a.y[(size_t)t * d + m] = acc;
        }
      }
    }
  }
}

}  // namespace

// host side --------------------------------------------------------------------
namespace {
struct FusedPlan {
  uint32_t c_rows, n_chunks, n_stages, stage_bytes;
  size_t smem;
};

bool fused_plan(const Ctx &c, FusedPlan *fp) {
  const moe_desc &D = c.desc;
  if (c.T < 1 || c.T > (uint32_t)kMaxT) return false;
  if (D.routed_fmt != MOE_FMT_Q8_0) return false;
  if (D.flags & (MOE_FLAG_DEBUG_TAPS | MOE_FLAG_FORCE_GEMV)) return false;
  if (D.flags & MOE_FLAG_FORCE_TC) return false;
  if (D.d % 256 || D.f % 256 || D.f_shared % 256) return false;
  if (c.R > 64) return false;
  const uint32_t d = D.d, fmax = c.fmax;
  const size_t b_bytes = (size_t)kBFeat * 2 * (d + d / 16);
  const uint32_t row_c = fmax + fmax / 16;
  uint32_t c_rows = (uint32_t)(b_bytes / row_c) / 8 * 8;
  if (c_rows == 0) return false;
  if (c_rows > d) c_rows = d;
  const size_t stage = ((b_bytes > (size_t)c_rows * row_c ? b_bytes : (size_t)c_rows * row_c) +
                        127) / 128 * 128;
  const size_t rest = (size_t)kMaxT * d + (size_t)kMaxT * (d / 32) * 4 + (size_t)kMaxT * fmax +
                      (size_t)kMaxT * (fmax / 32) * 4 + kMaxT * kBItemFeat * 4 +
                      kMaxStages * sizeof(StageDesc) + 2 * kMaxStages * 8 + 16 + 64 * 4 +
                      64 * 4 + 128;
  int dev = 0, max_smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
      cudaSuccess)
    return false;
  if ((size_t)max_smem < rest + 2 * stage) return false;
  uint32_t ns = (uint32_t)(((size_t)max_smem - rest) / stage);
  if (ns > (uint32_t)kMaxStages) ns = kMaxStages;
  fp->c_rows = c_rows;
  fp->n_chunks = (d + c_rows - 1) / c_rows;
  fp->n_stages = ns;
  fp->stage_bytes = (uint32_t)stage;
  fp->smem = rest + ns * stage;
  return true;
}
}  // namespace

size_t fused_sync_ints(const moe_desc *d) { return 4 + (size_t)d->n_expert + 1 + (size_t)d->d / 8; }

// counters start at zero every call; the error word is cleared with them
cudaError_t zero_decode_fused(const Ctx &c) {
  cudaError_t e = cudaMemsetAsync(c.ws + c.L.sync, 0, fused_sync_ints(&c.desc) * 4, c.stream);
  if (e != cudaSuccess) return e;
  return cudaMemsetAsync(c.ws + c.L.err, 0, 4, c.stream);
}

bool fused_eligible(const Ctx &c) {
  FusedPlan fp;
  return fused_plan(c, &fp);
}

cudaError_t launch_decode_fused(const Ctx &c, const float *x, const float *logits,
                                const float *bias, float *y) {
  FusedPlan fp;
  if (!fused_plan(c, &fp)) return cudaErrorNotSupported;
  const moe_desc &D = c.desc;
  FusedArgs a;
  a.E = D.n_expert;
  a.k = D.top_k;
  a.d = D.d;
  a.f = D.f;
  a.fs = D.f_shared;
  a.T = c.T;
  a.R = c.R;
  a.fmax = c.fmax;
  a.s = D.s;
  a.x = x;
  a.logits = logits;
  a.bias = bias;
  a.gq = (const int8_t *)c.wts.gate.q;
  a.uq = (const int8_t *)c.wts.up.q;
  a.dq = (const int8_t *)c.wts.down.q;
  a.gs = c.wts.gate.scale;
  a.us = c.wts.up.scale;
  a.ds = c.wts.down.scale;
  a.sgq = (const int8_t *)c.wts.s_gate.q;
  a.suq = (const int8_t *)c.wts.s_up.q;
  a.sdq = (const int8_t *)c.wts.s_down.q;
  a.sgs = c.wts.s_gate.scale;
  a.sus = c.wts.s_up.scale;
  a.sds = c.wts.s_down.scale;
  a.y = y;
  a.idx = (int32_t *)(c.ws + c.L.idx);
  a.w = (float *)(c.ws + c.L.w);
  a.off = (int32_t *)(c.ws + c.L.off);
  a.perm = (int32_t *)(c.ws + c.L.perm);
  a.pos = (int32_t *)(c.ws + c.L.pos);
  a.xq = (int8_t *)(c.ws + c.L.xq);
  a.xs = (float *)(c.ws + c.L.xs);
  a.hq = (int8_t *)(c.ws + c.L.hq);
  a.hs = (float *)(c.ws + c.L.hs);
  a.o = (float *)(c.ws + c.L.o);
  a.plan = (int *)(c.ws + c.L.plan);
  a.sync = (uint32_t *)(c.ws + c.L.sync);
  a.err = (uint32_t *)(c.ws + c.L.err);
  a.c_rows = fp.c_rows;
  a.n_chunks = fp.n_chunks;
  a.n_stages = fp.n_stages;
  a.stage_bytes = fp.stage_bytes;
  a.stall_test = (D.flags & MOE_FLAG_TEST_STALL) ? 1 : 0;
  a.wait_cycles = a.stall_test ? kStallTestCycles : kWaitCycles;
  cudaError_t e = cudaFuncSetAttribute(k_decode_fused, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)fp.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)c.sm_count);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = fp.smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode_fused, a);
}

}  // namespace moe
