// expert_tc.cu -- grouped expert FFN on the 5th-generation tensor cores (tcgen05),
// for experts with enough rows to make the FFN a real dense contraction (batch
// prefill: each layer's chunk-wide union of experts read once for many tokens,
// NeutronStar README, section "Long-prompt prefill").
//
// sm_103a has no int8 tcgen05 MMA, so the int8 codes travel as fp16 (every int8
// value is exact in fp16) through tcgen05.mma kind::f16 with fp32 accumulation.
// A 32-element block's dot product of int8 values is an integer of magnitude
// <= 32*127*127 < 2^24, exact in fp32, so each block gets its own TMEM
// accumulator; an epilogue reads it back (tcgen05.ld), applies the weight and
// activation block scales and sums the blocks in fp32 -- the same int32 block
// dots as the dp4a path.
//
// One CTA per SM loops over tiles of (expert, 128 output features, 64 rows).
// Warp roles:
//   0      TMA producer: int8 weight tile [128 x 64 B] per matrix into a staging
//          buffer, fp16 activation tile [64 x 64] (128B-swizzled) for the MMA
//   1      TMEM owner and MMA issuer (one thread)
//   2..5   converters: staging int8 -> fp16 in the K-major 128B-swizzle layout
//   6..13  epilogue: warps 6..9 take rows 0..31 of the tile, 10..13 rows 32..63;
//          warp w reads TMEM lanes 32*(w%4).. (= features)
// MAT = 2: gate and up, epilogue h = silu(g)*u requantised per 32 features;
// MAT = 1: down, epilogue o.
#include <cuda.h>
#include <string.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;  // features per tile (TMEM lanes)
constexpr int kBN = 64;   // rows per tile (MMA N)
constexpr int kBK = 64;   // K per stage (two 32-blocks)
constexpr int kTcThreads = 14 * 32;
constexpr int kEpiWarps = 8;
constexpr long long kTcWaitCycles = 4000000000ll;  // ~2 s
constexpr int kTcSpinIters = 1 << 26;
constexpr int kSuspendNs = 20000;  // try_wait suspend-time hint: waiting warps sleep, not spin

struct TcArgs {
  uint32_t E, d, f, fs, R, fmax, nb_in;  // nb_in: 32-blocks along K
  uint32_t K;                            // reduction length (d or f)
  uint32_t ws_row_stride;                // scales per weight row (= K / 32)
  const uint16_t *ws[2];                 // routed weight scales per matrix
  const uint16_t *sws[2];                // shared expert weight scales
  const float *xs;                       // activation block scales [slots][K/32]
  uint32_t xs_stride;                    // floats per slot row of xs
  const int *plan;
  int8_t *hq;                            // MAT=2: outputs
  float *hs;
  __half *hperm;                         // MAT=2: fp16 copy of the h codes [slots][fmax]
  float *o;                              // MAT=1: output [slots][d]
  int32_t *tap;                          // taps (null when off)
  uint32_t tap_nb;                       // blocks per tap row
  uint32_t *err;
  uint32_t n_stages, stage_bytes;
};

struct TcMaps {
  CUtensorMap w[2];   // routed weights, [E * rows][K] int8
  CUtensorMap sw[2];  // shared expert weights, [rows][K] int8
  CUtensorMap act;    // activations, [slots][K] fp16, 128B swizzle
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t s32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void bar_init(uint64_t *b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(s32(b)), "r"(n));
}
__device__ __forceinline__ void bar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(s32(b)) : "memory");
}
__device__ __forceinline__ void bar_expect(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s32(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool bar_wait(uint64_t *b, uint32_t parity) {
  const long long t0 = clock64();
  for (int i = 0; i < kTcSpinIters; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(s32(b)), "r"(parity), "n"(kSuspendNs)
        : "memory");
    if (done) return true;
    if (clock64() - t0 > kTcWaitCycles) return false;
  }
  return false;
}
__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, int x, int y,
                                       uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(s32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(s32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, fp16 inputs, fp32 accumulate
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          s32(bar))
      : "memory");
}
// 32 consecutive fp32 columns of this warp's 32 TMEM lanes
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// shared-memory matrix descriptor: K-major operand in the 128-byte swizzle
// layout (8-row groups of 1024 bytes), version 1
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t desc = 0;
  desc |= (uint64_t)((saddr >> 4) & 0x3FFF);
  desc |= (uint64_t)1 << 16;               // leading byte offset (unused for this layout)
  desc |= (uint64_t)(1024 >> 4) << 32;     // stride byte offset: next 8-row group
  desc |= (uint64_t)1 << 46;               // descriptor version
  desc |= (uint64_t)2 << 61;               // 128-byte swizzle
  return desc;
}

// instruction descriptor: D f32, A and B f16, both K-major, M = 128, N = kBN
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);

// int8 x4 -> two half2, exact: bias to 0..255, place under exponent 2^10, subtract 1152
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, 0x5140);
  hi = __byte_perm(u, 0x64646464u, 0x7362);
  const __half2 k = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  __half2 a = __hsub2(*reinterpret_cast<__half2 *>(&lo), k);
  __half2 b = __hsub2(*reinterpret_cast<__half2 *>(&hi), k);
  lo = *reinterpret_cast<uint32_t *>(&a);
  hi = *reinterpret_cast<uint32_t *>(&b);
}

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 3, %0;" ::"n"(kEpiWarps * 32) : "memory");
}

// tile list of the plan: v -> (expert, slot0, rows); tile t -> (v, m-tile, n-tile)
struct TcTile {
  int e, slot0, rows, m0, n0;
  bool ok;
};

template <int MAT>
__device__ __forceinline__ TcTile tc_tile(const PlanView &P, const TcArgs &a, int tile) {
  TcTile t;
  t.ok = false;
  const int U = P.hdr[5];
  const int *prefix = MAT == 2 ? P.tc_tile_gu : P.tc_tile_dn;
  int lo = 0, hi = U;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= tile) lo = mid; else hi = mid;
  }
  const int v = lo;
  t.e = P.tc_e[v];
  t.slot0 = P.tc_row0[v];
  t.rows = P.tc_rows[v];
  const int ntiles = (t.rows + kBN - 1) / kBN;
  const int local = tile - prefix[v];
  t.m0 = (local / ntiles) * kBM;
  t.n0 = (local % ntiles) * kBN;
  t.ok = true;
  return t;
}

template <int MAT, bool TAPS>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_expert_tc(const TcArgs a, const __grid_constant__ TcMaps maps) {
  extern __shared__ __align__(1024) uint8_t tsm_raw[];
  // 1024-byte alignment for the swizzled operands
  uint8_t *tsm = (uint8_t *)(((uintptr_t)tsm_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t NS = a.n_stages;
  PlanView P(const_cast<int *>(a.plan), a.E);
  const int total = MAT == 2 ? P.hdr[6] : P.hdr[7];
  const uint32_t KS = a.K / kBK;  // stages per tile
  // stage layout: [A16 mat0 16K][A16 mat1 16K][B 8K][A8 mat0 8K][A8 mat1 8K]
  constexpr uint32_t kA16 = kBM * kBK * 2, kB16 = kBN * kBK * 2, kA8 = kBM * kBK;
  uint8_t *ctrl = tsm + (size_t)NS * a.stage_bytes;
  uint64_t *ld_full = (uint64_t *)ctrl;          // [NS]
  uint64_t *a_ready = ld_full + 8;               // [NS]
  uint64_t *st_empty = a_ready + 8;              // [NS]
  uint64_t *d_full = st_empty + 8;               // [2]
  uint64_t *d_empty = d_full + 2;                // [2]
  uint32_t *tmem_holder = (uint32_t *)(d_empty + 2);
  volatile int *abort_flag = (volatile int *)(tmem_holder + 1);
  float *xs_stage = (float *)(tmem_holder + 4);  // [2 buffers][2 blocks][kBN]
  const uint32_t tmem_cols = MAT == 2 ? 512 : 256;

  if (tid == 0) {
    for (uint32_t i = 0; i < NS; ++i) {
      bar_init(&ld_full[i], 1);
      bar_init(&a_ready[i], 4);
      bar_init(&st_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      bar_init(&d_full[i], 1);
      bar_init(&d_empty[i], kEpiWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     s32(tmem_holder)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ============================ TMA producer
    if (lane == 0) {
      uint32_t g = 0;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
        const TcTile t = tc_tile<MAT>(P, a, tile);
        const bool sh = t.e == (int)a.E;
        const int wrow = sh ? t.m0 : (int)(t.e * (MAT == 2 ? (int)a.f : (int)a.d)) + t.m0;
        for (uint32_t ks = 0; ks < KS; ++ks, ++g) {
          const uint32_t s = g % NS, use = g / NS;
          if (use > 0 && !bar_wait(&st_empty[s], (use - 1) & 1u)) {
            atomicOr(a.err, kErrTimeout);
            *abort_flag = 1;
            break;
          }
          uint8_t *st = tsm + (size_t)s * a.stage_bytes;
          bar_expect(&ld_full[s], MAT * kA8 + kB16);
          for (int mi = 0; mi < MAT; ++mi)
            tma_2d(st + 2 * kA16 + kB16 + mi * kA8, sh ? &maps.sw[mi] : &maps.w[mi],
                   (int)(ks * kBK), wrow, &ld_full[s]);
          tma_2d(st + 2 * kA16, &maps.act, (int)(ks * kBK), t.slot0 + t.n0, &ld_full[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer
    if (lane == 0) {
      uint32_t g = 0, dbuf_use[2] = {0, 0};
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
        for (uint32_t ks = 0; ks < KS; ++ks, ++g) {
          const uint32_t s = g % NS, use = g / NS, b = g & 1u;
          bool ok = bar_wait(&a_ready[s], use & 1u);
          if (ok && dbuf_use[b] > 0) ok = bar_wait(&d_empty[b], (dbuf_use[b] - 1) & 1u);
          if (!ok) {
            atomicOr(a.err, kErrTimeout);
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          uint8_t *st = tsm + (size_t)s * a.stage_bytes;
          const uint32_t b_addr = s32(st + 2 * kA16);
#pragma unroll
          for (int blk = 0; blk < 2; ++blk)
#pragma unroll
            for (int mi = 0; mi < MAT; ++mi)
#pragma unroll
              for (int k16 = 0; k16 < 2; ++k16) {
                const uint32_t koff = (uint32_t)(blk * 2 + k16) * 32;  // bytes along K
                const uint64_t ad = sw128_desc(s32(st + mi * kA16) + koff);
                const uint64_t bd = sw128_desc(b_addr + koff);
                const uint32_t dcol = tmem + b * (tmem_cols / 2) + (uint32_t)(mi * 2 + blk) * kBN;
                tc_mma(dcol, ad, bd, kIdesc, k16 > 0);
              }
          tc_commit(&st_empty[s]);
          tc_commit(&d_full[b]);
          ++dbuf_use[b];
        }
      }
    }
  } else if (warp < 6) {
    // ============================ converters: row r = tid - 64 of the tile
    const int r = tid - 64;
    uint32_t g = 0;
    for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
      for (uint32_t ks = 0; ks < KS; ++ks, ++g) {
        const uint32_t s = g % NS, use = g / NS;
        if (!bar_wait(&ld_full[s], use & 1u)) {
          atomicOr(a.err, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        uint8_t *st = tsm + (size_t)s * a.stage_bytes;
        for (int mi = 0; mi < MAT; ++mi) {
          const uint4 *src = (const uint4 *)(st + 2 * kA16 + kB16 + mi * kA8 + r * kBK);
          uint8_t *dst_row = st + mi * kA16 + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // 16 int8 -> two 16-byte fp16 chunks
            const uint4 w = src[q];
            uint4 c0, c1;
            i8x4_to_h2x2(w.x, c0.x, c0.y);
            i8x4_to_h2x2(w.y, c0.z, c0.w);
            i8x4_to_h2x2(w.z, c1.x, c1.y);
            i8x4_to_h2x2(w.w, c1.z, c1.w);
            const int j0 = 2 * q, j1 = 2 * q + 1;  // 16-byte chunk index along K
            *(uint4 *)(dst_row + ((j0 ^ (r & 7)) << 4)) = c0;
            *(uint4 *)(dst_row + ((j1 ^ (r & 7)) << 4)) = c1;
          }
        }
        // generic-proxy writes become visible to the tensor core
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) bar_arrive(&a_ready[s]);
      }
    }
  } else {
    // ============================ epilogue
    const int ew = warp - 6;                    // 0..7
    const int quarter = warp & 3;               // TMEM lane quarter this warp may read
    const int half = ew >> 2;                   // rows [32*half, 32*half+32) of the tile
    const int et = ew * 32 + lane;              // 0..255
    const int feat = quarter * 32 + lane;       // feature within the tile (TMEM lane)
    uint32_t g = 0, dbuf_use[2] = {0, 0};
    for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
      const TcTile t = tc_tile<MAT>(P, a, tile);
      const bool sh = t.e == (int)a.E;
      const int width = MAT == 2 ? (int)(sh ? a.fs : a.f) : (int)a.d;
      const int wrow = (sh ? 0 : t.e * width) + t.m0 + feat;  // weight row of this feature
      float acc[MAT][32];
#pragma unroll
      for (int mi = 0; mi < MAT; ++mi)
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[mi][j] = 0.0f;
      int jt = -1;  // tapped feature index of this thread, if any
      if (TAPS) {
        const int wf = t.m0 + feat;
#pragma unroll
        for (int j = kNTap - 1; j >= 0; --j)
          if ((int)tap_feature(j, width) == wf) jt = j;
      }
      // scales of stage ks are loaded one stage ahead (registers), so their
      // latency hides behind the previous stage's drain
      const int pblk = et / kBN, pn = et % kBN;
      const bool prow = et < 2 * kBN && t.n0 + pn < t.rows;
      const float *pxs = a.xs + (size_t)(t.slot0 + t.n0 + pn) * a.xs_stride + pblk;
      const uint16_t *pws[MAT];
#pragma unroll
      for (int mi = 0; mi < MAT; ++mi)
        pws[mi] = (sh ? a.sws[mi] : a.ws[mi]) + (size_t)wrow * a.ws_row_stride;
      float nx_xs = prow ? __ldg(pxs) : 0.0f;
      uint32_t nx_ws[MAT];
#pragma unroll
      for (int mi = 0; mi < MAT; ++mi) nx_ws[mi] = __ldg((const uint32_t *)pws[mi]);
      for (uint32_t ks = 0; ks < KS; ++ks, ++g) {
        const uint32_t b = g & 1u;
        // activation scales of this stage's two blocks for the tile's 64 rows
        float *xsb = xs_stage + (size_t)(g & 1u) * 2 * kBN;
        if (et < 2 * kBN) xsb[pblk * kBN + pn] = nx_xs;
        float wsc[MAT][2];
#pragma unroll
        for (int mi = 0; mi < MAT; ++mi) {
          wsc[mi][0] = half_bits_to_float((uint16_t)(nx_ws[mi] & 0xFFFFu));
          wsc[mi][1] = half_bits_to_float((uint16_t)(nx_ws[mi] >> 16));
        }
        if (ks + 1 < KS) {
          nx_xs = prow ? __ldg(pxs + (ks + 1) * 2) : 0.0f;
#pragma unroll
          for (int mi = 0; mi < MAT; ++mi)
            nx_ws[mi] = __ldg((const uint32_t *)(pws[mi] + (ks + 1) * 2));
        }
        epi_sync();
        if (!bar_wait(&d_full[b], dbuf_use[b] & 1u)) {
          atomicOr(a.err, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int blk = 0; blk < 2; ++blk)
#pragma unroll
          for (int mi = 0; mi < MAT; ++mi) {
            float v[32];
            const uint32_t col = b * (tmem_cols / 2) + (uint32_t)(mi * 2 + blk) * kBN + half * 32;
            tc_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + col, v);
            const float* xsr = xsb + blk * kBN + half * 32;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              acc[mi][j] = __fmaf_rn(v[j], wsc[mi][blk] * xsr[j], acc[mi][j]);
            if (TAPS && jt >= 0) {
              const uint32_t kb = ks * 2 + blk;
              for (int j = 0; j < 32; ++j) {
                const int n = half * 32 + j;
                if (t.n0 + n < t.rows) {
                  const size_t slot = (size_t)(t.slot0 + t.n0 + n);
                  const size_t base = MAT == 2 ? ((slot * 2 + mi) * kNTap + jt) * a.tap_nb
                                               : (slot * kNTap + jt) * a.tap_nb;
                  a.tap[base + kb] = (int32_t)v[j];
                }
              }
            }
          }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) bar_arrive(&d_empty[b]);
        ++dbuf_use[b];
      }
      if (*abort_flag) break;
      // ---- tile output
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int n = half * 32 + j;
        const bool live = t.n0 + n < t.rows;
        const size_t slot = (size_t)(t.slot0 + t.n0 + n);
        if (MAT == 2) {
          // h = silu(g)*u, requantised over this warp's 32 consecutive features
          const float gv = acc[0][j], uv = acc[MAT - 1][j];
          const float h = __fmul_rn(__fdiv_rn(gv, __fadd_rn(1.0f, spec_exp(-gv))), uv);
          float amax = fabsf(h);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          const float sc = __fdiv_rn(amax, 127.0f);
          const int q = quant_one(h, sc);
          if (live) {
            const size_t fo = (size_t)t.m0 + feat;
            a.hq[slot * a.fmax + fo] = (int8_t)q;
            a.hperm[slot * a.fmax + fo] = __int2half_rn(q);
            if (lane == 0) a.hs[slot * (a.fmax / 32) + fo / 32] = sc;
          }
        } else {
          if (live) a.o[slot * a.d + t.m0 + feat] = acc[0][j];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(tmem_cols)
                 : "memory");
  }
}

// activations for the tensor path: fp16 copy of x codes in slot order
__global__ void __launch_bounds__(256)
    k_perm_x(const int8_t *__restrict__ xq, const int32_t *__restrict__ perm, uint32_t R,
             uint32_t slots, uint32_t k, uint32_t d, __half *__restrict__ xperm) {
  const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;  // 8-element chunks
  const uint64_t chunks = (uint64_t)slots * (d / 8);
  if (i >= chunks) return;
  const uint32_t slot = (uint32_t)(i / (d / 8)), c = (uint32_t)(i % (d / 8));
  const uint32_t t = slot < R ? (uint32_t)perm[slot] / k : slot - R;
  const uint2 w = *(const uint2 *)(xq + (size_t)t * d + 8 * c);
  uint4 out;
  i8x4_to_h2x2(w.x, out.x, out.y);
  i8x4_to_h2x2(w.y, out.z, out.w);
  *(uint4 *)(xperm + (size_t)slot * d + 8 * c) = out;
}

// activation scales in slot order
__global__ void __launch_bounds__(256)
    k_perm_xs(const float *__restrict__ xs, const int32_t *__restrict__ perm, uint32_t R,
              uint32_t slots, uint32_t k, uint32_t nb, float *__restrict__ xsperm) {
  const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (uint64_t)slots * nb) return;
  const uint32_t slot = (uint32_t)(i / nb), b = (uint32_t)(i % nb);
  const uint32_t t = slot < R ? (uint32_t)perm[slot] / k : slot - R;
  xsperm[i] = xs[(size_t)t * nb + b];
}

// ---------------------------------------------------------------- host
typedef CUresult (*EncodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiled)p;
  }
  return fn;
}

bool make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t cols,
              uint64_t rows, uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows,
              CUtensorMapSwizzle sw) {
  EncodeTiled fn = encode_fn();
  if (!fn || !base) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MAT, bool TAPS>
cudaError_t run_tc(const Ctx &c, const TcArgs &a, const TcMaps &maps, size_t smem) {
  auto kern = k_expert_tc<MAT, TAPS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<c.sm_count, kTcThreads, smem, c.stream>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace

bool tc_supported(const moe_desc &D) {
  if (D.routed_fmt != MOE_FMT_Q8_0) return false;
  if (D.d % 128 || D.f % 128 || (D.f_shared && D.f_shared % 128)) return false;
  return encode_fn() != nullptr;
}

// can any expert of a T-token call land on the tensor path (workspace sizing)?
bool tc_possible(const moe_desc &D, uint32_t T) {
  if (D.flags & MOE_FLAG_FORCE_GEMV) return false;
  if (D.routed_fmt != MOE_FMT_Q8_0) return false;
  if (D.d % 128 || D.f % 128 || (D.f_shared && D.f_shared % 128)) return false;
  return (D.flags & MOE_FLAG_FORCE_TC) ? T > 0 : T > kTcMinRows;
}

cudaError_t launch_tc_prepare(const Ctx &c, const int32_t *perm) {
  const uint32_t slots = c.R + (c.desc.f_shared ? c.T : 0);
  const uint64_t n1 = (uint64_t)slots * (c.desc.d / 8);
  if (n1 == 0) return cudaSuccess;
  k_perm_x<<<(unsigned)((n1 + 255) / 256), 256, 0, c.stream>>>(
      (const int8_t *)(c.ws + c.L.xq), perm, c.R, slots, c.desc.top_k, c.desc.d,
      (__half *)(c.ws + c.L.xperm));
  const uint64_t n2 = (uint64_t)slots * (c.desc.d / 32);
  k_perm_xs<<<(unsigned)((n2 + 255) / 256), 256, 0, c.stream>>>(
      (const float *)(c.ws + c.L.xs), perm, c.R, slots, c.desc.top_k, c.desc.d / 32,
      (float *)(c.ws + c.L.xsperm));
  return cudaGetLastError();
}

cudaError_t launch_tc(const Ctx &c, int mat) {
  const moe_desc &D = c.desc;
  const uint32_t slots = c.R + (D.f_shared ? c.T : 0);
  if (slots == 0) return cudaSuccess;
  TcArgs a;
  memset(&a, 0, sizeof a);
  TcMaps maps;
  memset(&maps, 0, sizeof maps);
  a.E = D.n_expert;
  a.d = D.d;
  a.f = D.f;
  a.fs = D.f_shared;
  a.R = c.R;
  a.fmax = c.fmax;
  a.plan = (const int *)(c.ws + c.L.plan);
  a.err = (uint32_t *)(c.ws + c.L.err);
  const bool taps = (D.flags & MOE_FLAG_DEBUG_TAPS) != 0;
  bool ok = true;
  if (mat == 2) {
    a.K = D.d;
    a.ws[0] = c.wts.gate.scale;
    a.ws[1] = c.wts.up.scale;
    a.sws[0] = c.wts.s_gate.scale;
    a.sws[1] = c.wts.s_up.scale;
    a.xs = (const float *)(c.ws + c.L.xsperm);
    a.xs_stride = D.d / 32;
    a.hq = (int8_t *)(c.ws + c.L.hq);
    a.hs = (float *)(c.ws + c.L.hs);
    a.hperm = (__half *)(c.ws + c.L.hperm);
    a.tap = taps ? (int32_t *)(c.ws + c.L.tap_gu) : nullptr;
    a.tap_nb = D.d / 32;
    ok &= make_map(&maps.w[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, c.wts.gate.q, D.d,
                   (uint64_t)D.n_expert * D.f, D.d, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    ok &= make_map(&maps.w[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, c.wts.up.q, D.d,
                   (uint64_t)D.n_expert * D.f, D.d, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (D.f_shared) {
      ok &= make_map(&maps.sw[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, c.wts.s_gate.q, D.d, D.f_shared,
                     D.d, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
      ok &= make_map(&maps.sw[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, c.wts.s_up.q, D.d, D.f_shared,
                     D.d, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
      maps.sw[0] = maps.w[0];
      maps.sw[1] = maps.w[1];
    }
    ok &= make_map(&maps.act, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, c.ws + c.L.xperm, D.d, slots,
                   (uint64_t)D.d * 2, kBK, kBN, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    a.K = D.f;  // the shared expert is on this path only when f_shared == f
    a.ws[0] = c.wts.down.scale;
    a.sws[0] = c.wts.s_down.scale;
    a.xs = (const float *)(c.ws + c.L.hs);
    a.xs_stride = c.fmax / 32;
    a.o = (float *)(c.ws + c.L.o);
    a.tap = taps ? (int32_t *)(c.ws + c.L.tap_dn) : nullptr;
    a.tap_nb = c.fmax / 32;
    ok &= make_map(&maps.w[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, c.wts.down.q, D.f,
                   (uint64_t)D.n_expert * D.d, D.f, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (D.f_shared)
      ok &= make_map(&maps.sw[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, c.wts.s_down.q, D.f_shared,
                     D.d, D.f_shared, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    else
      maps.sw[0] = maps.w[0];
    maps.w[1] = maps.w[0];
    maps.sw[1] = maps.sw[0];
    ok &= make_map(&maps.act, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, c.ws + c.L.hperm, c.fmax, slots,
                   (uint64_t)c.fmax * 2, kBK, kBN, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!ok) return cudaErrorInvalidValue;
  a.ws_row_stride = a.K / 32;
  a.nb_in = a.K / 32;
  const uint32_t stage = mat == 2 ? (2 * 16384 + 8192 + 2 * 8192) : (2 * 16384 + 8192 + 2 * 8192);
  a.stage_bytes = stage;
  a.n_stages = mat == 2 ? 3 : 3;
  const size_t smem = 1024 + (size_t)a.n_stages * stage + 2048;
  if (mat == 2)
    return taps ? run_tc<2, true>(c, a, maps, smem) : run_tc<2, false>(c, a, maps, smem);
  return taps ? run_tc<1, true>(c, a, maps, smem) : run_tc<1, false>(c, a, maps, smem);
}

}  // namespace moe
