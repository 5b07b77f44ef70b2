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
// RFMT: format of the routed experts' weights.  2-bit routed weights (code c in
// {0..3} meaning 2c - 3) are decoded by the converters into fp16 as exactly as
// int8 codes are, so the MMA computes the same exact integer block dots.  4-bit
// e2m1 routed weights go to the tensor cores as they are: tcgen05.mma
// kind::f8f6f4 with A = e2m1 (the converters only spread the packed codes into
// the operand layout: 16 codes in the first 8 bytes of each 16-byte chunk) and
// B = e4m3, the activation codes q carried as the two exact e4m3 digits of
// 2q = 32 hi + 2 lo (hi = floor(q/16) in [-8, 7], lo in [0, 15]), one MMA per
// digit into the same accumulator: the block dot sum(v * 2q) = sum(2v * q), the
// same exact integer as for the other formats (the block-dot taps check it).
// The shared expert is always Q8_0.
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
constexpr uint32_t kSG = 4;        // stages per scale group (8 blocks: a 16-byte fp16 box row)
constexpr uint32_t kScSlots = 3;   // scale groups in flight
// a scale slot: weight scales [MAT<=2][kBM rows][8] fp16 + activation scales [kBN rows][8] fp32
constexpr uint32_t kScSlotBytes = 2 * kBM * kSG * 2 * 2 + kBN * kSG * 2 * 4;
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
  const int32_t *eslot;  // expert -> weight slot (moe_weights.expert_slot), or null
  float routed_wmul;     // factor of the routed weight scales (0.5: e2m1 dots are of 2v)
  uint32_t *queue;       // [0] tiles taken, [1] CTAs done (fixed head, zero between calls)
  uint32_t n_stages, stage_bytes;
  unsigned long long *trace;  // MOE_FLAG_TRACE: kTcTraceWords per CTA, else null
};

// MOE_FLAG_TRACE words per CTA (cycles), gate/up at 0.., down at 8..
enum : int {
  kTcTrProdWaitEmpty = 0,  // producer waiting for a free stage
  kTcTrMmaWaitA = 1,       // MMA issuer waiting for converted operands
  kTcTrMmaWaitD = 2,       // MMA issuer waiting for a free accumulator buffer
  kTcTrCvtWaitFull = 3,    // converters waiting for the TMA data
  kTcTrEpiWaitD = 4,       // epilogue waiting for accumulators
  kTcTrEpiOut = 5,         // epilogue writing tile outputs
  kTcTrTotal = 6,          // kernel cycles (thread 0)
  kTcTrStages = 7,         // stages processed
  kTcTraceStride = 28      // words per CTA in the trace region
};

struct TcMaps {
  CUtensorMap w[2];    // routed weights, [E * rows][K] int8
  CUtensorMap sw[2];   // shared expert weights, [rows][K] int8
  CUtensorMap act;     // activations, [slots][K] fp16, 128B swizzle
  CUtensorMap ws[2];   // routed weight scales, [E * rows][K/32] fp16, box 8 x 128
  CUtensorMap sws[2];  // shared expert weight scales, [rows][K/32] fp16, box 8 x 128
  CUtensorMap xs;      // activation scales, [slots][K/32] fp32, box 8 x 64
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
// The MMA and commit helpers are called by a whole converged warp with
// warp-uniform operands; one lane (elect.sync) issues.  Timed on this part, a
// gate/up stage's 8 MMAs and its commit issued this way took ~680 cycles
// against ~890 from one lane of a divergent branch.
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, fp16 inputs, fp32 accumulate
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred e, p;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
// kind::f8f6f4: A e2m1, B e4m3, D f32
__device__ __forceinline__ void tc_mma_f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred e, p;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(
          s32(bar))
      : "memory");
}
// 16 consecutive fp32 columns of this warp's 32 TMEM lanes, no wait (tc_wait_ld)
__device__ __forceinline__ void tc_ld16_issue(uint32_t taddr, float (&v)[16]) {
  uint32_t *r = reinterpret_cast<uint32_t *>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
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

// instruction descriptor: D f32 (bit 4), A and B f16 (bits 7-9, 10-12: 0), both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24
constexpr uint32_t kIdescBase = (1u << 4) | ((uint32_t)(kBM >> 4) << 24);
__device__ __forceinline__ uint32_t idesc_for(uint32_t n) { return kIdescBase | ((n >> 3) << 17); }
// kind::f8f6f4: A e2m1 (5), B e4m3 (0)
__device__ __forceinline__ uint32_t idesc_f4_for(uint32_t n) {
  return idesc_for(n) | (5u << 7) | (0u << 10);
}

// The e4m3 byte of an integer v with at most 4 significant bits and |v| <= 256
// (exactly representable): sign, biased exponent floor(log2 |v|) + 7, the 3
// bits below the leading one.
__device__ __forceinline__ uint32_t e4m3_of_int(int v) {
  if (v == 0) return 0u;
  const uint32_t a = (uint32_t)(v < 0 ? -v : v);
  const int e = 31 - __clz((int)a);
  return (v < 0 ? 0x80u : 0u) | ((uint32_t)(e + 7) << 3) | (((a << 3) >> e) & 7u);
}
// the two e4m3 digits of 2q for an int8 code q: 32 hi and 2 lo, hi = floor(q/16)
__device__ __forceinline__ void e4m3_digits(int q, uint32_t &dhi, uint32_t &dlo) {
  const int hi = q >> 4;  // floor(q / 16), -8 .. 7
  dhi = e4m3_of_int(32 * hi);
  dlo = e4m3_of_int(2 * (q - 16 * hi));
}

// MMA width of a tile: its live rows rounded up to 16 (the MMA's N step at M = 128)
__device__ __forceinline__ int tile_cols(int rows, int n0) {
  const int live = min(kBN, rows - n0);
  return (live + 15) & ~15;
}

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

// 16 2-bit codes (byte b: codes 4b..4b+3, LSB first) -> eight half2 of 2c - 3,
// in K order: out[2b] = codes (4b, 4b+1), out[2b+1] = codes (4b+2, 4b+3).
// t_i holds code 4b+i in the low bits of byte b, under 0x3C; a byte permute puts
// each code's byte (0x3C | c) above a zero byte (the sign-replicated 0x3C|c),
// which is the fp16 1 + c/4; then 8 * (1 + c/4) - 11 = 2c - 3, exact.
__device__ __forceinline__ void q2x16_to_h2x8(uint32_t w, uint32_t (&out)[8]) {
  uint32_t t[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) t[i] = ((w >> (2 * i)) & 0x03030303u) | 0x3C3C3C3Cu;
  const __half2 k8 = __halves2half2(__ushort_as_half(0x4800), __ushort_as_half(0x4800));   // 8
  const __half2 km11 = __halves2half2(__ushort_as_half(0xC980), __ushort_as_half(0xC980));  // -11
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    // bytes: [sign(t_lo.b) = 0, t_lo.b, sign(t_hi.b) = 0, t_hi.b]
    const uint32_t sel = (8u | b) | ((uint32_t)b << 4) | ((8u | b) << 8) | ((4u + b) << 12);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t v = prmt_sx(t[2 * h], t[2 * h + 1], sel);
      __half2 r = __hfma2(*reinterpret_cast<__half2 *>(&v), k8, km11);
      out[2 * b + h] = *reinterpret_cast<uint32_t *>(&r);
    }
  }
}

// the two epilogue warps that read TMEM lane quarter q (one of each half) meet at
// named barrier 4 + q; they alone share rows of the split-K partial sums
__device__ __forceinline__ void epi_pair_sync(int quarter) {
  asm volatile("bar.sync %0, 64;" ::"r"(4 + quarter) : "memory");
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

// Tiles go out from a queue: the producer takes the CTA's next tile from a
// counter in the workspace's fixed head (the plan lists the widest, costliest
// tiles first) and publishes it to the CTA's other roles in a ring of
// kTileRing entries, each with an mbarrier of count 1 (a tile >= the total
// ends every role's loop).  The roles lag the producer by a few tiles at most
// (every tile has K/64 >= 4 stages, and the stage and accumulator rings hold
// fewer than 3 tiles' worth), so an entry is read before it is written again.
constexpr int kTileRing = 8;

// Stage geometry of a tile: MMA width ncol = live rows rounded up to 16, and
// gstages = stages whose accumulators share one TMEM buffer (ncol * gstages =
// kBN, so a buffer is always MAT * 2 * kBN columns).  The epilogue waits, reads
// and releases once per buffer instead of once per stage.
struct TileGeom {
  int ncol, gstages;
};
__device__ __forceinline__ TileGeom tile_geom(int rows, int n0) {
  TileGeom g;
  const int c = tile_cols(rows, n0);
  g.ncol = c <= 16 ? 16 : c <= 32 ? 32 : kBN;
  g.gstages = kBN / g.ncol;
  return g;
}
// TMEM column of (stage-in-buffer si, matrix mi, block bi) in buffer b
template <int MAT>
__device__ __forceinline__ uint32_t acc_col(uint32_t b, uint32_t half_cols, int si, int mi, int bi,
                                            int ncol) {
  return b * half_cols + (uint32_t)(((si * MAT + mi) * 2 + bi) * ncol);
}

// Epilogue of one tile.  NCM: columns per warp (16 or 32).  SPLIT (ncol <= 32):
// warp half h takes the K blocks of parity h over all columns, the halves'
// partial sums meeting in shared memory at the tile end; !SPLIT (ncol = 64):
// half h takes columns [32h, 32h + 32) of both blocks.  Warp w reads TMEM lanes
// 32*(w%4).. (= features).  Per block: acc += dot * (w-scale * x-scale), the
// scales coming from the scale ring (one slot per kSG stages, filled by TMA).
struct EpiState {
  uint32_t tmem, KS;
  uint32_t bufs, scgroups;  // accumulator buffers / scale groups consumed so far
  uint64_t *d_full;         // the control block's other barriers, the scale ring and
                            // the abort flag sit at fixed offsets from it
  float *red;
  long long t_wait, t_out;
};

template <int MAT, bool TAPS, int NCM, bool SPLIT, int RFMT>
__device__ __noinline__ void epi_tile(const TcArgs &a, EpiState &c, const TcTile &t,
                                      const TileGeom &geo) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ew = warp - 6;               // 0..7
  const int quarter = warp & 3;          // TMEM lane quarter this warp may read
  const int half = ew >> 2;
  const int feat = quarter * 32 + lane;  // feature within the tile (TMEM lane)
  const bool sh = t.e == (int)a.E;
  const int width = MAT == 2 ? (int)(sh ? a.fs : a.f) : (int)a.d;
  const float wmul = sh ? 1.0f : a.routed_wmul;  // exact (a power of two)
  const int col0 = SPLIT ? 0 : 32 * half;
  // accumulator pairs (columns 2i, 2i+1): the scale products and FMAs run as
  // packed fp32x2 operations, each lane rounded as the scalar operation would be
  float2 acc2[MAT][NCM / 2];
#define ACC(mi, j) (((j) & 1) ? acc2[mi][(j) >> 1].y : acc2[mi][(j) >> 1].x)
#pragma unroll
  for (int mi = 0; mi < MAT; ++mi)
#pragma unroll
    for (int j = 0; j < NCM / 2; ++j) acc2[mi][j] = make_float2(0.0f, 0.0f);
  int jt = -1;  // tapped feature index of this thread, if any
  if (TAPS) {
    const int wf = t.m0 + feat;
#pragma unroll
    for (int j = kNTap - 1; j >= 0; --j)
      if ((int)tap_feature(j, width) == wf) jt = j;
  }
  // The loop's counters and the TMEM base in registers for the whole tile (a
  // reference into the caller's frame is reloaded from local memory after
  // every asm with a memory clobber); the barriers, the scale ring and the
  // abort flag are fixed offsets from one base (the kernel's control block).
  const uint32_t KS = c.KS, tmem = c.tmem;
  constexpr uint32_t half_cols = MAT == 2 ? 256 : 128;
  uint32_t bufs = c.bufs, scgroups = c.scgroups;
  uint64_t *const d_full = c.d_full;
  uint64_t *const d_empty = d_full + 2;
  uint64_t *const sc_full = d_empty + 2;
  uint64_t *const sc_empty = sc_full + kScSlots;
  const uint8_t *const sc_ring = (const uint8_t *)(d_full - 24) - kScSlots * kScSlotBytes;
  volatile int *const abort_flag = (volatile int *)((uint32_t *)(sc_empty + kScSlots) + 1);
  long long t_wait = c.t_wait;
  for (uint32_t ks0 = 0; ks0 < KS; ks0 += geo.gstages) {
    const uint32_t b = bufs & 1u;
    const long long tw = clock64();
    if (!bar_wait(&d_full[b], (bufs >> 1) & 1u)) {
      atomicOr(a.err, kErrTimeout);
      *abort_flag = 1;
      c.bufs = bufs, c.scgroups = scgroups, c.t_wait = t_wait;
      return;
    }
    t_wait += clock64() - tw;
    tc_fence_after();
    const uint32_t nst = min((uint32_t)geo.gstages, KS - ks0);
    for (uint32_t si = 0; si < nst; ++si) {
      const uint32_t ks = ks0 + si;
      const uint32_t q = scgroups % kScSlots;  // scale slot of stage ks
      if (ks % kSG == 0) {
        if (!bar_wait(&sc_full[q], (scgroups / kScSlots) & 1u)) {
          atomicOr(a.err, kErrTimeout);
          *abort_flag = 1;
          c.bufs = bufs, c.scgroups = scgroups, c.t_wait = t_wait;
          return;
        }
      }
      const uint8_t *slot = sc_ring + (size_t)q * kScSlotBytes;
      const uint16_t *wsl = (const uint16_t *)slot;                       // [MAT][kBM][8]
      const float *xsl = (const float *)(slot + MAT * kBM * kSG * 2 * 2);  // [kBN][8]
      const uint32_t blk0 = (ks % kSG) * 2;  // first block of this stage in the slot
      float wsc[MAT][2];
#pragma unroll
      for (int mi = 0; mi < MAT; ++mi) {
        const uint32_t pair =
            *reinterpret_cast<const uint32_t *>(wsl + ((size_t)mi * kBM + feat) * 8 + blk0);
        wsc[mi][0] = half_bits_to_float((uint16_t)(pair & 0xFFFFu)) * wmul;
        wsc[mi][1] = half_bits_to_float((uint16_t)(pair >> 16)) * wmul;
      }
#pragma unroll
      for (int bi = 0; bi < 2; ++bi) {
        if (SPLIT && bi != half) continue;  // warp-uniform
#pragma unroll
        for (int c16 = 0; c16 < NCM / 16; ++c16) {
          // both matrices' 16 columns in flight together, one wait
          float v[MAT][16];
#pragma unroll
          for (int mi = 0; mi < MAT; ++mi)
            tc_ld16_issue(tmem + ((uint32_t)(quarter * 32) << 16) +
                              acc_col<MAT>(b, half_cols, (int)si, mi, bi, geo.ncol) + col0 +
                              16 * c16,
                          v[mi]);
          float xsv[16];  // the 16 rows' x scales of this block (shared by both matrices)
#pragma unroll
          for (int j = 0; j < 16; ++j) xsv[j] = xsl[(col0 + 16 * c16 + j) * 8 + blk0 + bi];
          tc_wait_ld();
#pragma unroll
          for (int mi = 0; mi < MAT; ++mi) {
            const float ws_b = wsc[mi][bi];
            const float2 ws2 = make_float2(ws_b, ws_b);
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              const float2 sc2 = __fmul2_rn(ws2, make_float2(xsv[j], xsv[j + 1]));
              float2 &a2 = acc2[mi][(16 * c16 + j) >> 1];
              a2 = __ffma2_rn(make_float2(v[mi][j], v[mi][j + 1]), sc2, a2);
            }
            if (TAPS && jt >= 0) {
              const uint32_t kb = ks * 2 + bi;
              for (int j = 0; j < 16; ++j) {
                const int n = col0 + 16 * c16 + j;
                if (t.n0 + n < t.rows) {
                  const size_t sl = (size_t)(t.slot0 + t.n0 + n);
                  const size_t base = MAT == 2 ? ((sl * 2 + mi) * kNTap + jt) * a.tap_nb
                                               : (sl * kNTap + jt) * a.tap_nb;
                  a.tap[base + kb] = (int32_t)v[mi][j];
                }
              }
            }
          }
        }
      }
      if (ks % kSG == kSG - 1 || ks + 1 == KS) {  // the scale slot's last stage
        __syncwarp();
        if (lane == 0) bar_arrive(&sc_empty[q]);
        ++scgroups;
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) bar_arrive(&d_empty[b]);
    ++bufs;
  }
  c.bufs = bufs;
  c.scgroups = scgroups;
  c.t_wait = t_wait;
  const long long t_o = clock64();
  if (SPLIT) {
    // odd blocks' partial sums (half 1) join the even blocks' (half 0)
    if (half == 1) {
#pragma unroll
      for (int mi = 0; mi < MAT; ++mi)
#pragma unroll
        for (int j = 0; j < NCM; ++j) c.red[((size_t)mi * kBM + feat) * 33 + j] = ACC(mi, j);
    }
    epi_pair_sync(quarter);
    if (half == 0) {
#pragma unroll
      for (int mi = 0; mi < MAT; ++mi)
#pragma unroll
        for (int j = 0; j < NCM; ++j)
          ACC(mi, j) = __fadd_rn(ACC(mi, j), c.red[((size_t)mi * kBM + feat) * 33 + j]);
    }
  }
  // ---- tile output: this warp's columns (half 0 only when split)
  if (!SPLIT || half == 0) {
#pragma unroll
    for (int j = 0; j < NCM; ++j) {
      const int n = col0 + j;
      if (t.n0 + n >= t.rows) break;  // warp-uniform: the tile's live rows end here
      const size_t sl = (size_t)(t.slot0 + t.n0 + n);
      if (MAT == 2) {
        // h = silu(g)*u, requantised over this warp's 32 consecutive features
        const float gv = ACC(0, j), uv = ACC(MAT - 1, j);
        const float h = __fmul_rn(__fdiv_rn(gv, __fadd_rn(1.0f, spec_exp(-gv))), uv);
        // |h| of finite values orders as its bit pattern: one warp max reduction
        const float amax =
            __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h))));
        const float sc = __fdiv_rn(amax, 127.0f);
        const int qv = quant_one(h, sc);
        const size_t fo = (size_t)t.m0 + feat;
        a.hq[sl * a.fmax + fo] = (int8_t)qv;
        if (RFMT == MOE_FMT_E2M1 && !sh) {
          // the down tiles' B operand: per 64-feature stage, the 32-hi digits of
          // 2q in the stage's first 64 bytes, the 2-lo digits in the next 64
          uint32_t dhi, dlo;
          e4m3_digits(qv, dhi, dlo);
          uint8_t *row = (uint8_t *)a.hperm + sl * a.fmax * 2 + (fo / 64) * 128 + fo % 64;
          row[0] = (uint8_t)dhi;
          row[64] = (uint8_t)dlo;
        } else {
          a.hperm[sl * a.fmax + fo] = __int2half_rn(qv);
        }
        if (lane == 0) a.hs[sl * (a.fmax / 32) + fo / 32] = sc;
      } else {
        a.o[sl * a.d + t.m0 + feat] = ACC(0, j);
      }
    }
  }
  if (SPLIT) epi_pair_sync(quarter);  // this quarter's red[] rows are free again
  c.t_out += clock64() - t_o;
}
#undef ACC

template <int MAT, bool TAPS, int RFMT>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_expert_tc(const TcArgs a, const __grid_constant__ TcMaps maps) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(1024) uint8_t tsm_raw[];
  // 1024-byte alignment for the swizzled operands
  uint8_t *tsm = (uint8_t *)(((uintptr_t)tsm_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t NS = a.n_stages;
  PlanView P(const_cast<int *>(a.plan), a.E);
  const int total = MAT == 2 ? P.hdr[6] : P.hdr[7];
  if (total == 0) return;  // no tensor-core tiles in this call's plan
  const uint32_t KS = a.K / kBK;  // stages per tile
  // stage layout: [A16 per matrix 16K][B 8K][A8 per matrix 8K]; a 2-bit or e2m1
  // tile stages its 16 or 32 code bytes per row at the start of each A8 area
  constexpr uint32_t kA16 = kBM * kBK * 2, kB16 = kBN * kBK * 2, kA8 = kBM * kBK;
  uint8_t *sc_ring = tsm + (size_t)NS * a.stage_bytes;  // [kScSlots][kScSlotBytes]
  uint8_t *ctrl = sc_ring + (size_t)kScSlots * kScSlotBytes;
  uint64_t *ld_full = (uint64_t *)ctrl;          // [NS]
  uint64_t *a_ready = ld_full + 8;               // [NS]
  uint64_t *st_empty = a_ready + 8;              // [NS]
  uint64_t *d_full = st_empty + 8;               // [2]
  uint64_t *d_empty = d_full + 2;                // [2]
  uint64_t *sc_full = d_empty + 2;               // [kScSlots]
  uint64_t *sc_empty = sc_full + kScSlots;       // [kScSlots]
  uint32_t *tmem_holder = (uint32_t *)(sc_empty + kScSlots);
  volatile int *abort_flag = (volatile int *)(tmem_holder + 1);
  volatile int *tile_ring = (volatile int *)(ctrl + 512);  // [kTileRing]
  uint64_t *tile_bar = (uint64_t *)(ctrl + 576);           // [kTileRing]
  float *red = (float *)(ctrl + 1024);  // [MAT][kBM features][33]: split-K partial sums
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
    for (uint32_t i = 0; i < kScSlots; ++i) {
      bar_init(&sc_full[i], 1);
      bar_init(&sc_empty[i], kEpiWarps);
    }
    for (int i = 0; i < kTileRing; ++i) bar_init(&tile_bar[i], 1);
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
  const long long t_start = clock64();
  long long t_wait0 = 0, t_wait1 = 0, t_out = 0;
  unsigned long long *tr =
      a.trace ? a.trace + (size_t)blockIdx.x * kTcTraceStride + (MAT == 2 ? 0 : 8) : nullptr;
  // round rd's tile, as the producer published it (total: none left)
  auto next_tile = [&](int rd) -> int {
    if (!bar_wait(&tile_bar[rd % kTileRing], (uint32_t)(rd / kTileRing) & 1u)) {
      atomicOr(a.err, kErrTimeout);
      *abort_flag = 1;
      return total;
    }
    return tile_ring[rd % kTileRing];
  };

  if (warp == 0) {
    // ============================ TMA producer: weights per stage, scales per kSG stages
    if (lane == 0) {
      uint32_t g = 0, scg = 0;
      for (int rd = 0; !*abort_flag; ++rd) {
        const int tile = (int)atomicAdd(a.queue, 1u);
        tile_ring[rd % kTileRing] = tile < total ? tile : total;
        bar_arrive(&tile_bar[rd % kTileRing]);
        if (tile >= total) break;
        const TcTile t = tc_tile<MAT>(P, a, tile);
        const bool sh = t.e == (int)a.E;
        // routed weights from the expert's slot (validated by k_plan)
        const int wrow =
            sh ? t.m0 : weight_slot(a.eslot, t.e) * (MAT == 2 ? (int)a.f : (int)a.d) + t.m0;
        for (uint32_t ks = 0; ks < KS; ++ks, ++g) {
          if (ks % kSG == 0) {
            // scales of stages ks .. ks+kSG-1: 8 blocks of the tile's weight rows
            // and activation rows
            const uint32_t q = scg % kScSlots, use = scg / kScSlots;
            const long long tw = clock64();
            const bool ok_s = use == 0 || bar_wait(&sc_empty[q], (use - 1) & 1u);
            t_wait0 += clock64() - tw;
            if (!ok_s) {
              atomicOr(a.err, kErrTimeout);
              *abort_flag = 1;
              break;
            }
            uint8_t *slot = sc_ring + (size_t)q * kScSlotBytes;
            bar_expect(&sc_full[q], MAT * kBM * kSG * 2 * 2 + kBN * kSG * 2 * 4);
            for (int mi = 0; mi < MAT; ++mi)
              tma_2d(slot + (size_t)mi * kBM * kSG * 2 * 2, sh ? &maps.sws[mi] : &maps.ws[mi],
                     (int)(ks * 2), wrow, &sc_full[q]);
            tma_2d(slot + MAT * kBM * kSG * 2 * 2, &maps.xs, (int)(ks * 2), t.slot0 + t.n0,
                   &sc_full[q]);
            ++scg;
          }
          const uint32_t s = g % NS, use = g / NS;
          const long long tw = clock64();
          const bool ok_e = use == 0 || bar_wait(&st_empty[s], (use - 1) & 1u);
          t_wait0 += clock64() - tw;
          if (!ok_e) {
            atomicOr(a.err, kErrTimeout);
            *abort_flag = 1;
            break;
          }
          uint8_t *st = tsm + (size_t)s * a.stage_bytes;
          // code bytes a row per stage: 64 (int8), 16 (2-bit), 32 (e2m1)
          const uint32_t rb = sh || RFMT == MOE_FMT_Q8_0 ? kBK
                              : RFMT == MOE_FMT_Q2S     ? kBK / 4
                                                        : kBK / 2;
          bar_expect(&ld_full[s], MAT * kBM * rb + kB16);
          for (int mi = 0; mi < MAT; ++mi)
            tma_2d(st + MAT * kA16 + kB16 + mi * kA8, sh ? &maps.sw[mi] : &maps.w[mi],
                   (int)(ks * rb), wrow, &ld_full[s]);
          tma_2d(st + MAT * kA16, &maps.act, (int)(ks * kBK), t.slot0 + t.n0, &ld_full[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer: a buffer holds gstages stages.  The
    // whole warp runs the loop (every lane waits, the results made warp-uniform),
    // and the MMAs and commits go out from one elected lane.
    uint32_t g = 0, bufs = 0;
    for (int rd = 0, tile; !*abort_flag && (tile = next_tile(rd)) < total; ++rd) {
      const TcTile tt = tc_tile<MAT>(P, a, tile);
      const TileGeom geo = tile_geom(tt.rows, tt.n0);
      // e2m1 routed tile: kind::f8f6f4 on the packed codes and the e4m3 digits
      const bool f4 = RFMT == MOE_FMT_E2M1 && tt.e != (int)a.E;
      const uint32_t idesc =
          f4 ? idesc_f4_for((uint32_t)geo.ncol) : idesc_for((uint32_t)geo.ncol);
      bool ok = true;
      for (uint32_t ks = 0; ks < KS; ++ks, ++g) {
        const uint32_t s = g % NS, use = g / NS, b = bufs & 1u;
        const uint32_t si = ks % (uint32_t)geo.gstages;
        const long long tw = clock64();
        ok = bar_wait(&a_ready[s], use & 1u);
        const long long tw2 = clock64();
        t_wait0 += tw2 - tw;
        if (ok && si == 0 && bufs >= 2) ok = bar_wait(&d_empty[b], ((bufs >> 1) - 1) & 1u);
        t_wait1 += clock64() - tw2;
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t *st = tsm + (size_t)s * a.stage_bytes;
        // descriptors of the stage's operands; offsets along K are added to the
        // address field (16-byte units; shared addresses stay below 2^18)
        const uint64_t a_desc = sw128_desc(s32(st));
        const uint64_t b_desc = sw128_desc(s32(st + MAT * kA16));
#pragma unroll
        for (int blk = 0; blk < 2; ++blk)
#pragma unroll
          for (int mi = 0; mi < MAT; ++mi) {
            const uint32_t dcol = tmem + acc_col<MAT>(b, tmem_cols / 2, (int)si, mi, blk,
                                                      geo.ncol);
            const uint64_t ad = a_desc + (uint64_t)(mi * (kA16 >> 4));
            if (f4) {
              // K = 32 a block: A chunks 2blk, 2blk+1; B's 32-hi digits in the
              // row's first 64 bytes, its 2-lo digits in the next 64
              tc_mma_f4(dcol, ad + 2u * blk, b_desc + 2u * blk, idesc, false);
              tc_mma_f4(dcol, ad + 2u * blk, b_desc + 4u + 2u * blk, idesc, true);
            } else {
#pragma unroll
              for (int k16 = 0; k16 < 2; ++k16) {
                const uint32_t kq = (uint32_t)(blk * 2 + k16) * 2;  // 32 bytes along K
                tc_mma(dcol, ad + kq, b_desc + kq, idesc, k16 > 0);
              }
            }
          }
        tc_commit(&st_empty[s]);
        if (si + 1 == (uint32_t)geo.gstages || ks + 1 == KS) {
          tc_commit(&d_full[b]);
          ++bufs;
        }
      }
      if (!ok) {
        if (lane == 0) atomicOr(a.err, kErrTimeout);
        *abort_flag = 1;
        break;
      }
    }
  } else if (warp < 6) {
    // ============================ converters: row r = tid - 64 of the tile
    const int r = tid - 64;
    uint32_t g = 0;
    for (int rd = 0, tile; !*abort_flag && (tile = next_tile(rd)) < total; ++rd) {
      // a 2-bit or e2m1 routed tile (the shared expert is Q8_0)
      const bool routed = RFMT != MOE_FMT_Q8_0 && tc_tile<MAT>(P, a, tile).e != (int)a.E;
      const bool q2 = RFMT == MOE_FMT_Q2S && routed;
      const bool f4 = RFMT == MOE_FMT_E2M1 && routed;
      for (uint32_t ks = 0; ks < KS; ++ks, ++g) {
        const uint32_t s = g % NS, use = g / NS;
        const long long tw = clock64();
        const bool ok_f = bar_wait(&ld_full[s], use & 1u);
        t_wait0 += clock64() - tw;
        if (!ok_f) {
          atomicOr(a.err, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        uint8_t *st = tsm + (size_t)s * a.stage_bytes;
        if (f4) {
          // row r's 32 code bytes = 64 e2m1 codes: codes 16j .. 16j+15 (8 bytes)
          // into the first half of 16-byte chunk j of the operand row, at
          // position j ^ (r&7) of its 128-byte swizzled row; the MMA reads
          // chunks 0..3 (K 0..63)
          for (int mi = 0; mi < MAT; ++mi) {
            const uint4 *src = (const uint4 *)(st + MAT * kA16 + kB16 + mi * kA8 + r * (kBK / 2));
            uint8_t *dst_row = st + mi * kA16 + (r >> 3) * 1024 + (r & 7) * 128;
            const uint4 c0 = src[0], c1 = src[1];
            *(uint4 *)(dst_row + ((0 ^ (r & 7)) << 4)) = make_uint4(c0.x, c0.y, 0u, 0u);
            *(uint4 *)(dst_row + ((1 ^ (r & 7)) << 4)) = make_uint4(c0.z, c0.w, 0u, 0u);
            *(uint4 *)(dst_row + ((2 ^ (r & 7)) << 4)) = make_uint4(c1.x, c1.y, 0u, 0u);
            *(uint4 *)(dst_row + ((3 ^ (r & 7)) << 4)) = make_uint4(c1.z, c1.w, 0u, 0u);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) bar_arrive(&a_ready[s]);
          continue;
        }
        if (q2) {
          // row r's 16 code bytes (rows 16 B apart: a quarter-warp reads 128
          // contiguous bytes) -> 8 fp16 chunks; chunk j lands at position
          // j ^ (r&7) of its swizzled row (distinct over a quarter-warp)
          for (int mi = 0; mi < MAT; ++mi) {
            const uint4 w = *(const uint4 *)(st + MAT * kA16 + kB16 + mi * kA8 + r * (kBK / 4));
            uint8_t *dst_row = st + mi * kA16 + (r >> 3) * 1024 + (r & 7) * 128;
            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int v = 0; v < 4; ++v) {  // codes 16v .. 16v+15 = chunks 2v, 2v+1
              uint32_t h[8];
              q2x16_to_h2x8(wv[v], h);
              const int j0 = 2 * v, j1 = 2 * v + 1;
              *(uint4 *)(dst_row + ((j0 ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
              *(uint4 *)(dst_row + ((j1 ^ (r & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) bar_arrive(&a_ready[s]);
          continue;
        }
        for (int mi = 0; mi < MAT; ++mi) {
          const uint4 *src = (const uint4 *)(st + MAT * kA16 + kB16 + mi * kA8 + r * kBK);
          uint8_t *dst_row = st + mi * kA16 + (r >> 3) * 1024 + (r & 7) * 128;
          // Chunk order per row pair s = (r/2)%4: q = qq ^ g(s), g = (0, 2, 3, 1).
          // Loads: the staging rows are 64 B apart, so in a quarter-warp (rows
          // r..r+7) even rows use 16-byte bank groups q and odd rows 4 + q:
          // distinct because g is a permutation.  Stores: chunk 2q (2q+1) lands
          // at position 2q ^ (r&7) of its 128-byte swizzled row, i.e. 2(q ^ s)
          // (+1): distinct because s -> g(s) ^ s is a permutation too.  Both are
          // conflict-free.
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {  // 16 int8 -> two 16-byte fp16 chunks
            const int q = qq ^ (int)((0x78u >> (2 * ((r >> 1) & 3))) & 3u);
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
    EpiState c;
    c.tmem = tmem;
    c.KS = KS;
    c.bufs = 0;
    c.scgroups = 0;
    c.d_full = d_full;
    c.red = red;
    c.t_wait = 0;
    c.t_out = 0;
    for (int rd = 0, tile; !*abort_flag && (tile = next_tile(rd)) < total; ++rd) {
      const TcTile t = tc_tile<MAT>(P, a, tile);
      const TileGeom geo = tile_geom(t.rows, t.n0);
      if (geo.ncol == 16) epi_tile<MAT, TAPS, 16, true, RFMT>(a, c, t, geo);
      else if (geo.ncol == 32) epi_tile<MAT, TAPS, 32, true, RFMT>(a, c, t, geo);
      else epi_tile<MAT, TAPS, 32, false, RFMT>(a, c, t, geo);
    }
    t_wait0 = c.t_wait;
    t_out = c.t_out;
  }
  if (warp == 0 && lane == 0) {
    // the last producer out zeroes the queue for the next call (every other
    // producer has taken its last tile before it counts itself out)
    __threadfence();
    if (atomicAdd(a.queue + 1, 1u) == gridDim.x - 1) {
      atomicExch(a.queue, 0u);
      atomicExch(a.queue + 1, 0u);
    }
  }
  if (tr && lane == 0) {
    if (warp == 0) tr[kTcTrProdWaitEmpty] = t_wait0;
    if (warp == 1) {
      tr[kTcTrMmaWaitA] = t_wait0;
      tr[kTcTrMmaWaitD] = t_wait1;
    }
    if (warp == 2) tr[kTcTrCvtWaitFull] = t_wait0;
    if (warp == 6) {
      tr[kTcTrEpiWaitD] = t_wait0;
      tr[kTcTrEpiOut] = t_out;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tr && threadIdx.x == 0) tr[kTcTrTotal] = clock64() - t_start;
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(tmem_cols)
                 : "memory");
  }
}

// activations for the tensor path in slot order (nothing when the plan sends no
// expert to the tensor cores): an fp16 copy of the x codes, or for the routed
// slots of an e2m1 layer (`digits`) the e4m3 digits of 2q, per 64-element
// stage 64 bytes of 32-hi digits then 64 of 2-lo digits (the same 128 bytes);
// and the x block scales in slot order (the thread of a block's first chunk)
__global__ void __launch_bounds__(256)
    k_perm_x(const int8_t *__restrict__ xq, const float *__restrict__ xs,
             const int32_t *__restrict__ perm, uint32_t R, uint32_t slots, uint32_t k,
             uint32_t d, const int *plan, uint32_t E, __half *__restrict__ xperm,
             float *__restrict__ xsperm, int digits) {
  pdl_trigger();
  pdl_wait();
  if (PlanView(const_cast<int *>(plan), E).hdr[5] == 0) return;
  const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;  // 8-element chunks
  const uint64_t chunks = (uint64_t)slots * (d / 8);
  if (i >= chunks) return;
  const uint32_t slot = (uint32_t)(i / (d / 8)), c = (uint32_t)(i % (d / 8));
  const uint32_t t = slot < R ? (uint32_t)perm[slot] / k : slot - R;
  if ((c & 3u) == 0) xsperm[(size_t)slot * (d / 32) + c / 4] = xs[(size_t)t * (d / 32) + c / 4];
  const uint2 w = *(const uint2 *)(xq + (size_t)t * d + 8 * c);
  if (digits && slot < R) {
    uint32_t hi[2] = {0u, 0u}, lo[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = (int)(int8_t)(((i < 4 ? w.x : w.y) >> (8 * (i & 3))) & 0xFFu);
      uint32_t dh, dl;
      e4m3_digits(q, dh, dl);
      hi[i >> 2] |= dh << (8 * (i & 3));
      lo[i >> 2] |= dl << (8 * (i & 3));
    }
    uint8_t *row = (uint8_t *)xperm + (size_t)slot * d * 2 + (8 * c / 64) * 128 + (8 * c) % 64;
    *(uint2 *)row = make_uint2(hi[0], hi[1]);
    *(uint2 *)(row + 64) = make_uint2(lo[0], lo[1]);
    return;
  }
  uint4 out;
  i8x4_to_h2x2(w.x, out.x, out.y);
  i8x4_to_h2x2(w.y, out.z, out.w);
  *(uint4 *)(xperm + (size_t)slot * d + 8 * c) = out;
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

template <int MAT, bool TAPS, int RFMT>
cudaError_t run_tc(const Ctx &c, const TcArgs &a, const TcMaps &maps, size_t smem) {
  auto kern = k_expert_tc<MAT, TAPS, RFMT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_k(kern, c.sm_count, kTcThreads, smem, c.stream, c.chained, a, maps);
  c.chained = true;
  return e;
}

}  // namespace

// the scale rows (K/32 fp16) of every matrix must be whole 16-byte TMA rows (and
// a 2-bit or e2m1 code row, K/4 or K/2 bytes, a multiple of 16 bytes: K % 256
// covers all)
bool tc_supported(const moe_desc &D) {
  if (D.routed_fmt != MOE_FMT_Q8_0 && D.routed_fmt != MOE_FMT_Q2S &&
      D.routed_fmt != MOE_FMT_E2M1)
    return false;
  if (D.d % 256 || D.f % 256 || (D.f_shared && D.f_shared % 256)) return false;
  return encode_fn() != nullptr;
}

bool tc_weights_aligned(const Ctx &c) {
  const moe_weights &w = c.wts;
  auto a16 = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
  bool ok = a16(w.gate.q) && a16(w.up.q) && a16(w.down.q) && a16(w.gate.scale) &&
            a16(w.up.scale) && a16(w.down.scale);
  if (c.desc.f_shared)
    ok = ok && a16(w.s_gate.q) && a16(w.s_up.q) && a16(w.s_down.q) && a16(w.s_gate.scale) &&
         a16(w.s_up.scale) && a16(w.s_down.scale);
  return ok;
}

// can any expert of a T-token call land on the tensor path (workspace sizing)?
bool tc_possible(const moe_desc &D, uint32_t T) {
  if (D.flags & MOE_FLAG_FORCE_GEMV) return false;
  if (D.routed_fmt != MOE_FMT_Q8_0 && D.routed_fmt != MOE_FMT_Q2S &&
      D.routed_fmt != MOE_FMT_E2M1)
    return false;
  if (D.d % 256 || D.f % 256 || (D.f_shared && D.f_shared % 256)) return false;
  // unforced, only from kTcMinTokens tokens: below that no expert brings enough
  // tiles to pay for the tensor kernels and their activation copies
  return (D.flags & MOE_FLAG_FORCE_TC) ? T > 0 : T >= kTcMinTokens && T > tc_min_rows_for(D.routed_fmt);
}

cudaError_t launch_tc_prepare(const Ctx &c, const int32_t *perm) {
  const uint32_t slots = c.R + (c.desc.f_shared ? c.T : 0);
  const uint64_t n1 = (uint64_t)slots * (c.desc.d / 8);
  if (n1 == 0) return cudaSuccess;
  const cudaError_t e =
      launch_k(k_perm_x, (unsigned)((n1 + 255) / 256), 256, 0, c.stream, c.chained,
               (const int8_t *)(c.ws + c.L.xq), (const float *)(c.ws + c.L.xs), perm, c.R, slots,
               c.desc.top_k, c.desc.d, (const int *)(c.ws + c.L.plan), c.desc.n_expert,
               (__half *)(c.ws + c.L.xperm), (float *)(c.ws + c.L.xsperm),
               c.desc.routed_fmt == MOE_FMT_E2M1 ? 1 : 0);
  c.chained = true;
  return e;
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
  a.eslot = c.wts.expert_slot;
  a.plan = (const int *)(c.ws + c.L.plan);
  a.err = (uint32_t *)(c.ws + c.L.err);
  a.queue = (uint32_t *)(c.ws + c.L.sync) + (mat == 2 ? kQueueTcGateup : kQueueTcDown);
  a.trace = (D.flags & MOE_FLAG_TRACE) && c.L.trace ? (unsigned long long *)(c.ws + c.L.trace)
                                                     : nullptr;
  const bool taps = (D.flags & MOE_FLAG_DEBUG_TAPS) != 0;
  const bool q2 = D.routed_fmt == MOE_FMT_Q2S;
  const bool f4 = D.routed_fmt == MOE_FMT_E2M1;
  // routed code planes: int8 [rows][K], box 64 x 128; 2-bit [rows][K/4] bytes,
  // box 16 x 128; e2m1 [rows][K/2] bytes, box 32 x 128
  const uint32_t qdiv = q2 ? 4 : f4 ? 2 : 1;
  a.routed_wmul = f4 ? 0.5f : 1.0f;
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
    ok &= make_map(&maps.w[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, c.wts.gate.q, D.d / qdiv,
                   (uint64_t)c.wexp * D.f, D.d / qdiv, kBK / qdiv, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    ok &= make_map(&maps.w[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, c.wts.up.q, D.d / qdiv,
                   (uint64_t)c.wexp * D.f, D.d / qdiv, kBK / qdiv, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
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
    // scales: 8 blocks (kSG stages) of 128 weight rows / 64 activation rows per copy
    ok &= make_map(&maps.ws[0], CU_TENSOR_MAP_DATA_TYPE_UINT16, c.wts.gate.scale, D.d / 32,
                   (uint64_t)c.wexp * D.f, D.d / 16, kSG * 2, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    ok &= make_map(&maps.ws[1], CU_TENSOR_MAP_DATA_TYPE_UINT16, c.wts.up.scale, D.d / 32,
                   (uint64_t)c.wexp * D.f, D.d / 16, kSG * 2, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (D.f_shared) {
      ok &= make_map(&maps.sws[0], CU_TENSOR_MAP_DATA_TYPE_UINT16, c.wts.s_gate.scale, D.d / 32,
                     D.f_shared, D.d / 16, kSG * 2, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
      ok &= make_map(&maps.sws[1], CU_TENSOR_MAP_DATA_TYPE_UINT16, c.wts.s_up.scale, D.d / 32,
                     D.f_shared, D.d / 16, kSG * 2, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
      maps.sws[0] = maps.ws[0];
      maps.sws[1] = maps.ws[1];
    }
    ok &= make_map(&maps.xs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, c.ws + c.L.xsperm, D.d / 32, slots,
                   (uint64_t)(D.d / 32) * 4, kSG * 2, kBN, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    a.K = D.f;  // the shared expert is on this path only when f_shared == f
    a.ws[0] = c.wts.down.scale;
    a.sws[0] = c.wts.s_down.scale;
    a.xs = (const float *)(c.ws + c.L.hs);
    a.xs_stride = c.fmax / 32;
    a.o = (float *)(c.ws + c.L.o);
    a.tap = taps ? (int32_t *)(c.ws + c.L.tap_dn) : nullptr;
    a.tap_nb = c.fmax / 32;
    ok &= make_map(&maps.w[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, c.wts.down.q, D.f / qdiv,
                   (uint64_t)c.wexp * D.d, D.f / qdiv, kBK / qdiv, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (D.f_shared)
      ok &= make_map(&maps.sw[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, c.wts.s_down.q, D.f_shared,
                     D.d, D.f_shared, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    else
      maps.sw[0] = maps.w[0];
    maps.w[1] = maps.w[0];
    maps.sw[1] = maps.sw[0];
    ok &= make_map(&maps.act, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, c.ws + c.L.hperm, c.fmax, slots,
                   (uint64_t)c.fmax * 2, kBK, kBN, CU_TENSOR_MAP_SWIZZLE_128B);
    ok &= make_map(&maps.ws[0], CU_TENSOR_MAP_DATA_TYPE_UINT16, c.wts.down.scale, D.f / 32,
                   (uint64_t)c.wexp * D.d, D.f / 16, kSG * 2, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (D.f_shared)
      ok &= make_map(&maps.sws[0], CU_TENSOR_MAP_DATA_TYPE_UINT16, c.wts.s_down.scale,
                     D.f_shared / 32, D.d, D.f_shared / 16, kSG * 2, kBM,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
    else
      maps.sws[0] = maps.ws[0];
    maps.ws[1] = maps.ws[0];
    maps.sws[1] = maps.sws[0];
    ok &= make_map(&maps.xs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, c.ws + c.L.hs, c.fmax / 32, slots,
                   (uint64_t)(c.fmax / 32) * 4, kSG * 2, kBN, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (!ok) return cudaErrorInvalidValue;
  a.ws_row_stride = a.K / 32;
  a.nb_in = a.K / 32;
  // stage: [fp16 A per matrix 16 KB][fp16 B 8 KB][int8 A per matrix 8 KB]
  const uint32_t stage = (uint32_t)mat * (16384 + 8192) + 8192;
  a.stage_bytes = stage;
  a.n_stages = mat == 2 ? 3 : 5;
  // alignment slack | stages | scale ring | barriers and flags | split-K partial sums
  const size_t smem = 1024 + (size_t)a.n_stages * stage + (size_t)kScSlots * kScSlotBytes + 1024 +
                      (size_t)mat * kBM * 33 * 4;
  if (q2) {
    if (mat == 2)
      return taps ? run_tc<2, true, MOE_FMT_Q2S>(c, a, maps, smem)
                  : run_tc<2, false, MOE_FMT_Q2S>(c, a, maps, smem);
    return taps ? run_tc<1, true, MOE_FMT_Q2S>(c, a, maps, smem)
                : run_tc<1, false, MOE_FMT_Q2S>(c, a, maps, smem);
  }
  if (f4) {
    if (mat == 2)
      return taps ? run_tc<2, true, MOE_FMT_E2M1>(c, a, maps, smem)
                  : run_tc<2, false, MOE_FMT_E2M1>(c, a, maps, smem);
    return taps ? run_tc<1, true, MOE_FMT_E2M1>(c, a, maps, smem)
                : run_tc<1, false, MOE_FMT_E2M1>(c, a, maps, smem);
  }
  if (mat == 2)
    return taps ? run_tc<2, true, MOE_FMT_Q8_0>(c, a, maps, smem)
                : run_tc<2, false, MOE_FMT_Q8_0>(c, a, maps, smem);
  return taps ? run_tc<1, true, MOE_FMT_Q8_0>(c, a, maps, smem)
              : run_tc<1, false, MOE_FMT_Q8_0>(c, a, maps, smem);
}

}  // namespace moe
