// expert_stream.cu -- dp4a expert FFN for small batches, the weights streamed
// into shared memory by the bulk-copy engine.
//
// The multi-kernel path's experts with few rows (every expert below 32 tokens a
// call, above it the experts with at most 6 rows, 4 for e2m1) are bound by the
// weight stream:
// each selected expert's rows are read once per call and applied to all of its
// rows (the union-of-experts read of NeutronStar README, "MTP speculative
// decoding"; the indexed per-expert FFN).  Rather than every warp loading its
// weight codes into registers (a few KB in flight per warp), one producer lane
// per CTA streams each work item's slice of one expert's weight rows with
// cp.async.bulk (one-CTA copies, no multicast) into a ring of four ~52 KB
// shared-memory stages, ~200 KB per SM in flight, and 12 consumer warps compute
// from shared memory with dp4a (the dp4a expert kernels of "What this branch
// adds over upstream").
//
//  * One CTA per SM, persistent; no CTA waits on another.  Work items go out
//    in chunks of 8 consecutive ones from a queue (a counter in the
//    workspace's fixed head that each CTA's producer takes chunks from), the
//    shared expert's first -- a row per token, its items cost the most -- then
//    the routed experts' (slices of one expert, mostly, whose activation rows
//    then stay in L1): hot experts' items (more rows, more passes) and the
//    shared expert's no longer leave some CTAs working long after the rest.
//    The last producer to finish zeroes the counter for the next call.
//  * The CTA's i-th item goes to stage i % 4 and is read by consumer group
//    i % 3 (4 warps), which learns the item from the stage header (an empty
//    header ends its loop).  Each group takes its items in order, and item i
//    waits only for item i - 4 to leave its stage, so the ring always moves.
//    13 warps: at most 4 on each of the SM's four sub-partitions, so a thread
//    may hold 128 registers.
//  * The stage's previous item i - 4 belongs to another group, so a group
//    reaching item i can find that item still in flight: its full barrier is
//    then two phases behind, where a parity wait would pass at once.  A
//    consumer therefore first waits for the release of item i - 4 (the empty
//    barrier, at most one phase behind: the producer issued item i - 4 only
//    after item i - 8 was released), then for item i's bytes.
//  * The producer looks one item ahead: the next item's plan lookup and its
//    first rows' tokens (the permutation) are in flight while it issues the
//    current item's copies, and each stage starts with a header (expert rows,
//    first output, the first rows' activation rows) that the consumers read
//    instead of repeating the lookup.
//  * Gate/up item: 4 consecutive Q8_0 features of one expert (16 of 2-bit or 8
//    of e2m1 routed weights, whose blocks a lane decodes once for every row),
//    their gate and up rows (codes + K/32 fp16 scales each).  The group's warps take a pair of
//    features over one K half each, for every row of the expert, in passes of
//    2 rows whose activation blocks they load at once; the halves' partial
//    sums meet in shared memory, summed in half order, and h = silu(g)*u goes
//    out in fp32; the requantisation kernel follows.
//  * Down item: 4*RW consecutive output rows of one expert's down matrix (Q8_0,
//    or 2-bit / e2m1 rows decoded a block at a time for both slots of a pass);
//    warp w takes RW of them against the h codes of every row (slot) of the
//    expert, in passes of 2 slots whose h blocks it loads at once.  For Q8_0
//    the producer first prefetches each new run of items' h rows into L1.
//  * Lane l holds whole 32-blocks l, l+32, ..: their exact int32 dots (the
//    block-dot taps) scaled by w-scale * x-scale into fp32 sums that meet in
//    the warp sum.  A block's two 16-byte halves are read from shared memory
//    in an order that keeps each quarter-warp on distinct banks.
//  * Every wait is bounded; on timeout the kernel flags kErrTimeout, stops
//    issuing, waits (bounded) for the copies it has in flight and exits.
#include <algorithm>

#include "stream_ptx.cuh"

namespace moe {
namespace {

constexpr int kStStages = 4;                           // shared-memory stages
constexpr int kStGroups = 3;                           // consumer groups
constexpr int kStGroupWarps = 4;                       // consumer warps per group
constexpr int kStConsWarps = kStGroups * kStGroupWarps;
constexpr int kStProdWarp = kStConsWarps;              // lane 0 issues the copies
constexpr int kStThreads = (kStConsWarps + 1) * 32;
constexpr int kStRows = 2;                             // activation rows per pass
constexpr int kHdrRows = 8;                            // rows whose activation row a header holds
constexpr long long kStWaitCycles = 4000000000ll;      // ~2 s at 2 GHz
constexpr uint32_t kStBarBytes = 128;                  // 11 mbarriers + the abort flag
constexpr uint32_t kStSmemMax = 227u * 1024u;          // opt-in dynamic shared memory a CTA
constexpr uint32_t kStHdrBytes = 64;                   // stage header
// gate/up partial sums: [group][2 pass parities][4 warps][8 values] fp32
constexpr int kGuVals = 2 * 2 * kStRows;  // gate/up x feature of the pair x row
// routed features per gate/up item by weight format: Q8_0 4, 2-bit 16, e2m1 8
// (stages of 35-52 KB at the layers' widths); the shared expert's items are
// always 4 Q8_0 features
template <int FMT>
__host__ __device__ constexpr int fpi_of() {
  return FMT == MOE_FMT_Q2S ? 16 : FMT == MOE_FMT_E2M1 ? 8 : 4;
}
constexpr int kGuValsMax = 2 * (16 / 2) * kStRows;  // the low-bit consumer's, 2-bit
constexpr uint32_t kStPartPerGroup = 2 * kStGroupWarps * kGuValsMax;  // floats
constexpr uint32_t kStPartFloats = kStGroups * kStPartPerGroup;
// largest stage: the dynamic shared memory of one CTA (227 KB) less the plan
// of a 1024-expert layer, the barriers and the partial sums, over the stages
constexpr uint32_t kStStageMax =
    (kStSmemMax - (uint32_t)(sizeof(int) * (4 * 1025 + 1)) - kStBarBytes - 4 * kStPartFloats) /
    kStStages / 16 * 16;
// x blocks per lane per row: K/64 blocks a half, d <= 6144 (Q8_0 items) or
// d <= 4096 (2-bit and e2m1 items: fewer registers beside their decoded blocks)
constexpr int kGuJ = 3;
constexpr int kGuJLowBit = 2;
// h blocks per lane per row and segment in the down stage
constexpr int kDnJ = 2;

struct StArgs {
  const int *plan;
  uint32_t E, k, d, f, fs, R;
  uint32_t K, Ks;             // reduction length of a routed / shared row
  uint32_t out_per_e;         // down: output rows per expert (d)
  const int8_t *q[2], *sq[2];        // routed / shared codes (gate/up: gate, up; down: down)
  const uint16_t *sc[2], *ssc[2];    // their block scales
  uint32_t rows_per_slot;     // routed weight rows per expert slot (gate/up: f; down: d)
  const int32_t *eslot;       // expert -> weight slot, or null
  const int8_t *act;          // activation codes: x [T][d] (gate/up), h [slots][fmax] (down)
  const int8_t *act_t;        // gate/up, 2-bit routed weights: x codes, 16-code groups transposed
  const float *act_s;         // their block scales
  uint32_t act_stride, act_s_stride;
  const int32_t *perm;        // gate/up: slot -> row (token = row / k)
  float *out;                 // gate/up: h [slots][out_stride]; down: o [slots][out_stride]
  uint32_t out_stride;
  int32_t *tap;               // MOE_FLAG_DEBUG_TAPS, else null
  uint32_t tap_nb;            // blocks per tap row
  uint32_t *err;
  uint32_t stage_bytes;
  uint32_t *queue;            // [0] chunks taken, [1] producers done (fixed head, zero between calls)
  unsigned long long *trace;  // MOE_FLAG_TRACE: this kernel's words of the trace region, else null
};



// MOE_FLAG_TRACE words per CTA (SM cycles), at kStTraceBase + (down ? kStTraceDown : 0)
// + CTA * kStTraceStride of the workspace's trace region
enum : int {
  kStTrProdWait = 0,    // producer waiting for a free stage
  kStTrItems = 1,       // items issued
  kStTrProdTotal = 2,   // producer: kernel entry to its last copy landed
  kStTrSetup = 3,       // kernel entry to the first copy issued
  kStTrConsWait = 4,    // + warp: consumer warp waiting for a full stage
  kStTrConsWork = 16,   // + warp: consumer warp computing
  kStTraceStride = 32,
  kStTraceBase = 16384,
  kStTraceDown = 8192,
  kStTraceCtas = 256
};

// stage header, written by the producer before it arms the stage's barrier
struct StageHdr {
  int row0, nrows, n0, sh;  // expert's first slot, its rows, first output, shared expert?
  int K;                    // reduction length
  int act_row[kHdrRows];    // gate/up: the tokens of its first rows
  int pad[3];
};
static_assert(sizeof(StageHdr) == kStHdrBytes, "stage header size");

// one work item: rows [n0, n0 + rows) of each of the MAT matrices of an expert
struct Item {
  int row0, nrows, n0;
  bool sh;
  int nf;      // weight rows of each matrix in the item
  uint32_t K;
  uint32_t rb;  // code bytes of one weight row
  const int8_t *q[2];
  const uint16_t *s[2];
};

// The call's items: the routed experts' first, then the shared expert's (the
// last expert of the plan's list, when it is there).  Gate/up: routed items of
// fpi_of<RFMT> features, shared items of 4 (Q8_0); down: NROWS output rows
// throughout, out_per_e / NROWS per expert.
struct ItemCount {
  int routed, items;
};
template <int MAT, int NROWS, int RFMT>
__device__ __forceinline__ ItemCount item_count(const StArgs &a, const SmemPlan &S, int U) {
  const bool shared = U > 0 && S.e[U - 1] == (int)a.E;
  ItemCount n;
  if (MAT == 2) {
    const int routed_feats = S.item[shared ? U - 1 : U];
    n.routed = routed_feats / fpi_of<RFMT>();
    n.items = n.routed + (shared ? (S.item[U] - routed_feats) / 4 : 0);
  } else {
    const int per = (int)(a.out_per_e / NROWS);
    n.routed = (shared ? U - 1 : U) * per;
    n.items = U * per;
  }
  return n;
}

template <int MAT, int NROWS, int RFMT>
__device__ __forceinline__ Item item_at(const StArgs &a, const SmemPlan &S, int U,
                                        const ItemCount &n, int g) {
  Item it;
  int u, n0;
  if (MAT == 2) {
    if (g < n.routed) {
      const int feat = g * fpi_of<RFMT>();
      u = find_slot(S.item, U, feat);
      n0 = feat - S.item[u];
      it.nf = fpi_of<RFMT>();
    } else {
      u = U - 1;
      n0 = (g - n.routed) * 4;
      it.nf = 4;
    }
  } else {
    const int per = (int)(a.out_per_e / NROWS);
    u = g / per;
    n0 = (g - u * per) * NROWS;
    it.nf = NROWS;
  }
  const int e = S.e[u];
  it.row0 = S.row0[u];
  it.nrows = S.rows[u];
  it.n0 = n0;
  it.sh = e == (int)a.E;
  it.K = it.sh ? a.Ks : a.K;
  it.rb = (uint32_t)row_bytes(it.sh ? MOE_FMT_Q8_0 : RFMT, it.K);
  // first weight row of the item in its matrix (k_plan validated the slot)
  const size_t r = it.sh ? (size_t)n0
                         : (size_t)weight_slot(a.eslot, e) * a.rows_per_slot + (size_t)n0;
#pragma unroll
  for (int m = 0; m < MAT; ++m) {
    it.q[m] = (it.sh ? a.sq[m] : a.q[m]) + r * it.rb;
    it.s[m] = (it.sh ? a.ssc[m] : a.sc[m]) + r * (it.K / 32);
  }
  return it;
}

// The call's items in the order a chunk queue hands them out: chunks of
// kChunk consecutive items, the shared expert's first (the costliest: a row per
// token), then the routed experts' (slices of one expert, mostly, whose
// activation rows then stay in L1).  Each CTA's producer takes the next chunk
// from a counter in the workspace's fixed head when it needs one, so the CTAs
// finish together whatever their items cost.
constexpr int kChunk = 8;
struct Chunks {
  int routed, items, n_shared, n;  // routed items, all items, shared chunks, chunks
  __device__ __forceinline__ int first(int c) const {
    return c < n_shared ? routed + c * kChunk : (c - n_shared) * kChunk;
  }
  __device__ __forceinline__ int end(int c) const {
    return c < n_shared ? min(routed + (c + 1) * kChunk, items)
                        : min((c - n_shared + 1) * kChunk, routed);
  }
};

__device__ __forceinline__ Chunks chunks_of(const ItemCount &n) {
  Chunks ch;
  ch.routed = n.routed;
  ch.items = n.items;
  ch.n_shared = (n.items - n.routed + kChunk - 1) / kChunk;
  ch.n = ch.n_shared + (n.routed + kChunk - 1) / kChunk;
  return ch;
}

// activation row of slot p: its token (gate/up: the shared expert's slots R..
// are the tokens in order, a routed slot's row comes from the permutation) or
// the slot itself (down: h rows are per slot)
template <int MAT>
__device__ __forceinline__ int act_row_of(const StArgs &a, bool sh, int p) {
  if (MAT == 1) return p;
  return sh ? p - (int)a.R : a.perm[p] / (int)a.k;
}

// N (16 or 32) values of every lane summed over the warp, transposed: on
// return lane l holds the warp total of value l % N (31 shuffles; a fixed order
// of fp32 adds)
template <int N>
__device__ __forceinline__ float transpose_sum(float (&v)[N], int lane) {
#pragma unroll
  for (int s = 16; s >= N; s >>= 1)
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], s);
#pragma unroll
  for (int s = N / 2; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = upper ? v[i] : v[i + s];
      const float keep = upper ? v[i + s] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return v[0];
}

// barrier of one consumer group's four warps: an mbarrier of count 4 (lane 0 of
// each warp arrives after a __syncwarp, so the warp's shared-memory writes are
// released), passed with a bounded wait on the phase of parity `par`
__device__ __forceinline__ bool group_sync(uint64_t *gbar, uint32_t par, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(gbar);
  return mbar_wait(gbar, par, kStWaitCycles);
}

// exact int32 dot of the 32-byte block at `w` (shared memory) with the
// activation block x.  The two 16-byte halves are read in the order `swap`
// (lanes with bit 2 set read the upper half first), so that a quarter-warp's
// eight 16-byte reads of eight consecutive blocks fall on distinct banks.
__device__ __forceinline__ int block_dot(const int8_t *w, const W8 &x, bool swap) {
  const uint4 a = lds16(w + (swap ? 16 : 0)), b = lds16(w + (swap ? 0 : 16));
  const uint4 xl = make_uint4(x.v[0], x.v[1], x.v[2], x.v[3]);
  const uint4 xh = make_uint4(x.v[4], x.v[5], x.v[6], x.v[7]);
  return dot16(a, swap ? xh : xl) + dot16(b, swap ? xl : xh);
}

// gate/up of the item's 4 features for every row of its expert.  Warp w takes
// features 2(w/2), 2(w/2)+1 over K half w%2; lane l holds whole 32-blocks
// l, l+32, .. of the half (at most 3 for d <= 6144).  A pass of 2 rows loads its
// activation blocks before any use.  Each lane's 8 partial sums (gate/up x
// feature x row) are summed over the warp, and the two halves of a feature in
// half order through shared memory (part: [2 pass parities][4 warps][8]); warp
// w then finishes feature 2(w/2) + w%2.  Stage layout after the header: gate
// codes [4][K], up codes [4][K], gate scales [4][K/32], up scales [4][K/32].
// Returns false if the group barrier's wait gave up.
template <bool TAPS>
__device__ __forceinline__ bool gateup_stage(const StArgs &a, const StageHdr &h,
                                             const int *hdr_rows, const uint8_t *w, int wi,
                                             int lane, float *part, uint64_t *gbar, uint32_t &par,
                                             uint64_t *empty_bar) {
  const uint32_t K = (uint32_t)h.K, nb = K / 32, nb2 = nb / 2;
  const int fp = wi >> 1, hk = wi & 1;  // feature pair, K half
  const int8_t *gcode = (const int8_t *)w;
  const int8_t *ucode = gcode + (size_t)kStGroupWarps * K;
  const uint16_t *gsc = (const uint16_t *)(w + (size_t)2 * kStGroupWarps * K);
  const uint16_t *usc = gsc + (size_t)kStGroupWarps * nb;
  const uint32_t width = h.sh ? a.fs : a.f;
  const bool swap = (lane >> 2) & 1;
  int jt[2];
#pragma unroll
  for (int f = 0; f < 2; ++f) jt[f] = TAPS ? tapped((uint32_t)(h.n0 + 2 * fp + f), width) : -1;
  for (int r0 = 0; r0 < h.nrows; r0 += kStRows) {
    const int nr = min(kStRows, h.nrows - r0);
    W8 xr[kStRows][kGuJ];
    float xsr[kStRows][kGuJ];
#pragma unroll
    for (int r = 0; r < kStRows; ++r) {
      const int rr = r0 + (r < nr ? r : 0);
      const int tok = rr < kHdrRows ? hdr_rows[rr] : act_row_of<2>(a, h.sh != 0, h.row0 + rr);
      const int8_t *xp = a.act + (size_t)tok * a.act_stride;
      const float *xsp = a.act_s + (size_t)tok * a.act_s_stride;
#pragma unroll
      for (int j = 0; j < kGuJ; ++j) {
        const uint32_t bl = lane + 32u * j, b = hk * nb2 + bl;
        const bool ok = r < nr && bl < nb2;
        if (ok) {
          xr[r][j] = ld_cached32(xp + 32 * b);
          xsr[r][j] = __ldg(xsp + b);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) xr[r][j].v[q] = 0u;
          xsr[r][j] = 0.0f;
        }
      }
    }
    float v[kGuVals];  // [m = gate, up][feature of the pair][row]
#pragma unroll
    for (int i = 0; i < kGuVals; ++i) v[i] = 0.0f;
    constexpr int kU = 2 * kStRows;  // offset of the up values
#pragma unroll
    for (int f = 0; f < 2; ++f) {
      const int fr = 2 * fp + f;  // feature row within the stage
#pragma unroll
      for (int j = 0; j < kGuJ; ++j) {
        const uint32_t bl = lane + 32u * j, b = hk * nb2 + bl;
        if (bl < nb2) {
          const float sg = half_bits_to_float(gsc[(size_t)fr * nb + b]);
          const float su = half_bits_to_float(usc[(size_t)fr * nb + b]);
#pragma unroll
          for (int r = 0; r < kStRows; ++r) {
            if (r < nr) {  // warp-uniform
              const int pg = block_dot(gcode + (size_t)fr * K + 32 * b, xr[r][j], swap);
              const int pu = block_dot(ucode + (size_t)fr * K + 32 * b, xr[r][j], swap);
              const int ig = f * kStRows + r;
              v[ig] = __fmaf_rn((float)pg, sg * xsr[r][j], v[ig]);
              v[kU + ig] = __fmaf_rn((float)pu, su * xsr[r][j], v[kU + ig]);
              if (TAPS && jt[f] >= 0) {
                int32_t *t = a.tap +
                             ((size_t)(h.row0 + r0 + r) * 2 * kNTap + (size_t)jt[f]) * a.tap_nb + b;
                t[0] = pg;
                t[(size_t)kNTap * a.tap_nb] = pu;
              }
            }
          }
        }
      }
    }
    // the stage is no longer read once its last pass has its dot products
    if (r0 + kStRows >= h.nrows) {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
    }
    const float tot = transpose_sum<kGuVals>(v, lane);
    float *pp = part + (size_t)par * kStGroupWarps * kGuVals;
    if (lane < kGuVals) pp[wi * kGuVals + lane] = tot;
    if (!group_sync(gbar, par, lane)) return false;
    // warp wi finishes feature 2 fp + hk: lane r < nr adds the K halves (half 0
    // first) of its gate and up values
    if (lane < nr) {
      const int ig = hk * kStRows + lane;
      const float *p0 = pp + (2 * fp) * kGuVals, *p1 = p0 + kGuVals;
      const float g = __fadd_rn(p0[ig], p1[ig]), u = __fadd_rn(p0[kU + ig], p1[kU + ig]);
      const float hv = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, spec_exp(-g))), u);
      a.out[(size_t)(h.row0 + r0 + lane) * a.out_stride + h.n0 + 2 * fp + hk] = hv;
    }
    par ^= 1u;
  }
  return true;
}

// gate/up of a routed item of 2-bit or e2m1 weights: fpi_of<RFMT> features
// (FP = half of them a warp pair) for every row of the expert.  Warp w takes
// features (w/2) FP .. + FP - 1 over K half w%2; lane l holds whole 32-blocks
// l, l+32, .. of the half: 8 code bytes (2-bit) or 16 (e2m1) from the stage,
// decoded once per block and dotted with every row's activation block (2-bit:
// activations 16-code-group transposed) -- the register GEMV's exact block
// dots.  The 2 FP x 2 partial sums of each lane are summed over the warp, the
// two K halves of a feature in half order through shared memory; warp w then
// finishes FP/2 features.  Stage layout after the header: gate codes
// [fpi][rb], up codes [fpi][rb], gate scales [fpi][K/32], up scales [fpi][K/32].
template <int RFMT, bool TAPS>
__device__ __forceinline__ bool gateup_stage_lb(const StArgs &a, const StageHdr &h,
                                                const int *hdr_rows, const uint8_t *w, int wi,
                                                int lane, float *part, uint64_t *gbar,
                                                uint32_t &par, uint64_t *empty_bar) {
  constexpr int FPI = fpi_of<RFMT>(), FP = FPI / 2;
  constexpr int NV = 2 * FP * kStRows;  // [m][feature of the pair][row]
  constexpr int BB = RFMT == MOE_FMT_Q2S ? 8 : 16;  // code bytes a block
  const uint32_t K = (uint32_t)h.K, nb = K / 32, nb2 = nb / 2, rb = nb * BB;
  const int fp = wi >> 1, hk = wi & 1;
  const int8_t *gcode = (const int8_t *)w;
  const int8_t *ucode = gcode + (size_t)FPI * rb;
  const uint16_t *gsc = (const uint16_t *)(w + (size_t)2 * FPI * rb);
  const uint16_t *usc = gsc + (size_t)FPI * nb;
  const int8_t *act = RFMT == MOE_FMT_Q2S ? a.act_t : a.act;
  int jt[FP];
#pragma unroll
  for (int f = 0; f < FP; ++f) jt[f] = TAPS ? tapped((uint32_t)(h.n0 + fp * FP + f), a.f) : -1;
  for (int r0 = 0; r0 < h.nrows; r0 += kStRows) {
    const int nr = min(kStRows, h.nrows - r0);
    W8 xr[kStRows][kGuJLowBit];
    float xsr[kStRows][kGuJLowBit];
    int sx[kStRows][kGuJLowBit];
#pragma unroll
    for (int r = 0; r < kStRows; ++r) {
      const int rr = r0 + (r < nr ? r : 0);
      const int tok = rr < kHdrRows ? hdr_rows[rr] : act_row_of<2>(a, false, h.row0 + rr);
      const int8_t *xp = act + (size_t)tok * a.act_stride;
      const float *xsp = a.act_s + (size_t)tok * a.act_s_stride;
#pragma unroll
      for (int j = 0; j < kGuJLowBit; ++j) {
        const uint32_t bl = lane + 32u * j, b = hk * nb2 + bl;
        if (r < nr && bl < nb2) {
          xr[r][j] = ld_cached32(xp + 32 * b);
          xsr[r][j] = __ldg(xsp + b);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) xr[r][j].v[q] = 0u;
          xsr[r][j] = 0.0f;
        }
        sx[r][j] = block_sum(xr[r][j]);
      }
    }
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = 0.0f;
    constexpr int kU = NV / 2;
#pragma unroll
    for (int f = 0; f < FP; ++f) {
      const int fr = fp * FP + f;  // feature row within the item
#pragma unroll
      for (int j = 0; j < kGuJLowBit; ++j) {
        const uint32_t bl = lane + 32u * j, b = hk * nb2 + bl;
        if (bl < nb2) {
#pragma unroll
          for (int m = 0; m < 2; ++m) {  // gate, then up: one decoded block live
            const uint16_t *scp = m == 0 ? gsc : usc;
            const int8_t *cp = (m == 0 ? gcode : ucode) + (size_t)fr * rb + BB * b;
            const float sw = half_bits_to_float(scp[(size_t)fr * nb + b]) * scale_mul<RFMT>();
            WBlock<RFMT> wb;
            if constexpr (RFMT == MOE_FMT_Q2S) wb.c = *(const uint2 *)cp;
            else wb.c = *(const uint4 *)cp;
            wb.prep();
#pragma unroll
            for (int r = 0; r < kStRows; ++r) {
              if (r < nr) {  // warp-uniform
                const int pd = wb.dot(xr[r][j], sx[r][j]);
                const int iv = m * kU + f * kStRows + r;
                v[iv] = __fmaf_rn((float)pd, sw * xsr[r][j], v[iv]);
                if (TAPS && jt[f] >= 0)
                  a.tap[(((size_t)(h.row0 + r0 + r) * 2 + m) * kNTap + (size_t)jt[f]) * a.tap_nb +
                        b] = pd;
              }
            }
          }
        }
      }
    }
    if (r0 + kStRows >= h.nrows) {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
    }
    const float tot = transpose_sum<NV>(v, lane);
    float *pp = part + (size_t)par * kStGroupWarps * NV;
    if (lane < NV) pp[wi * NV + lane] = tot;
    if (!group_sync(gbar, par, lane)) return false;
    // warp wi finishes features (wi/2) FP + (wi%2) FP/2 .. + FP/2 - 1: lane l
    // takes feature (wi%2) FP/2 + l/2 of the pair, row l%2
    const int fl = hk * (FP / 2) + (lane >> 1), r = lane & 1;
    if (lane < FP && r < nr) {
      const int ig = fl * kStRows + r;
      const float *p0 = pp + (2 * fp) * NV, *p1 = p0 + NV;
      const float g = __fadd_rn(p0[ig], p1[ig]), u = __fadd_rn(p0[kU + ig], p1[kU + ig]);
      const float hv = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, spec_exp(-g))), u);
      a.out[(size_t)(h.row0 + r0 + r) * a.out_stride + h.n0 + fp * FP + fl] = hv;
    }
    par ^= 1u;
  }
  return true;
}

// down rows n0 + wi*RW .. + RW - 1 for every row (slot) of the item's expert,
// in passes of 2 slots and segments of 32*kDnJ blocks (lane l: whole 32-blocks
// l, l+32, ..), every h block of a segment loaded before any use.  Stage layout
// after the header: codes [4*RW][K], scales [4*RW][K/32].  Arrives on the
// stage's empty barrier after its last read.
template <int RW, bool TAPS>
__device__ __forceinline__ void down_stage(const StArgs &a, const StageHdr &h, const uint8_t *w,
                                           int wi, int lane, uint64_t *empty_bar) {
  static_assert(RW * kStRows <= 16, "one transposed warp sum per pass");
  constexpr int kRows = kStGroupWarps * RW;
  const uint32_t K = (uint32_t)h.K, nb = K / 32;
  const int8_t *wc = (const int8_t *)w + (size_t)wi * RW * K;
  const uint16_t *wsc = (const uint16_t *)(w + (size_t)kRows * K) + (size_t)wi * RW * nb;
  const int m0 = h.n0 + wi * RW;
  const bool swap = (lane >> 2) & 1;
  int jt[RW];
#pragma unroll
  for (int q = 0; q < RW; ++q) jt[q] = TAPS ? tapped((uint32_t)(m0 + q), a.d) : -1;
  for (int r0 = 0; r0 < h.nrows; r0 += kStRows) {
    const int nr = min(kStRows, h.nrows - r0);
    int slot[kStRows];
    const int8_t *hp[kStRows];
    const float *hsp[kStRows];
#pragma unroll
    for (int r = 0; r < kStRows; ++r) {
      slot[r] = h.row0 + r0 + (r < nr ? r : 0);
      hp[r] = a.act + (size_t)slot[r] * a.act_stride;
      hsp[r] = a.act_s + (size_t)slot[r] * a.act_s_stride;
    }
    float v[16];  // [row q][slot r] at q * kStRows + r
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
#pragma unroll 1
    for (uint32_t b0 = 0; b0 < nb; b0 += 32 * kDnJ) {
      W8 hx[kStRows][kDnJ];
      float hsc[kStRows][kDnJ];
#pragma unroll
      for (int r = 0; r < kStRows; ++r)
#pragma unroll
        for (int j = 0; j < kDnJ; ++j) {
          const uint32_t b = b0 + lane + 32u * j;
          if (r < nr && b < nb) {
            hx[r][j] = ld_cached32(hp[r] + 32 * b);
            hsc[r][j] = __ldg(hsp[r] + b);
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) hx[r][j].v[q] = 0u;
            hsc[r][j] = 0.0f;
          }
        }
#pragma unroll
      for (int q = 0; q < RW; ++q)
#pragma unroll
        for (int j = 0; j < kDnJ; ++j) {
          const uint32_t b = b0 + lane + 32u * j;
          if (b < nb) {
            const float sw = half_bits_to_float(wsc[(size_t)q * nb + b]);
#pragma unroll
            for (int r = 0; r < kStRows; ++r) {
              if (r < nr) {
                const int p = block_dot(wc + (size_t)q * K + 32 * b, hx[r][j], swap);
                v[q * kStRows + r] = __fmaf_rn((float)p, sw * hsc[r][j], v[q * kStRows + r]);
                if (TAPS && jt[q] >= 0)
                  a.tap[((size_t)slot[r] * kNTap + (size_t)jt[q]) * a.tap_nb + b] = p;
              }
            }
          }
        }
    }
    if (r0 + kStRows >= h.nrows) {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
    }
    const float tot = transpose_sum<16>(v, lane);
    const int q = lane / kStRows, r = lane % kStRows;
    if (lane < 16 && q < RW && r < nr) a.out[(size_t)slot[r] * a.out_stride + m0 + q] = tot;
  }
}

// down rows n0 + wi*RW .. + RW - 1 of a routed item of 2-bit or e2m1 weights,
// for every slot of its expert, in passes of 2 slots and segments of 32*kDnJ
// blocks: lane l takes whole 32-blocks l, l+32, .., each row's block decoded
// once from the stage (8 or 16 code bytes) and dotted with both slots' h blocks
// (2-bit: h codes 16-code-group transposed) -- the register GEMV's exact block
// dots.  Stage layout after the header: codes [4*RW][rb], scales [4*RW][K/32].
// Arrives on the stage's empty barrier after its last read.
template <int RFMT, int RW, bool TAPS>
__device__ __forceinline__ void down_stage_lb(const StArgs &a, const StageHdr &h,
                                              const uint8_t *w, int wi, int lane,
                                              uint64_t *empty_bar) {
  static_assert(RW * kStRows <= 16, "one transposed warp sum per pass");
  constexpr int kRows = kStGroupWarps * RW;
  constexpr int BB = RFMT == MOE_FMT_Q2S ? 8 : 16;  // code bytes a block
  const uint32_t K = (uint32_t)h.K, nb = K / 32, rb = nb * BB;
  const int8_t *wc = (const int8_t *)w + (size_t)wi * RW * rb;
  const uint16_t *wsc = (const uint16_t *)(w + (size_t)kRows * rb) + (size_t)wi * RW * nb;
  const int8_t *act = RFMT == MOE_FMT_Q2S ? a.act_t : a.act;
  const int m0 = h.n0 + wi * RW;
  int jt[RW];
#pragma unroll
  for (int q = 0; q < RW; ++q) jt[q] = TAPS ? tapped((uint32_t)(m0 + q), a.d) : -1;
  for (int r0 = 0; r0 < h.nrows; r0 += kStRows) {
    const int nr = min(kStRows, h.nrows - r0);
    int slot[kStRows];
    const int8_t *hp[kStRows];
    const float *hsp[kStRows];
#pragma unroll
    for (int r = 0; r < kStRows; ++r) {
      slot[r] = h.row0 + r0 + (r < nr ? r : 0);
      hp[r] = act + (size_t)slot[r] * a.act_stride;
      hsp[r] = a.act_s + (size_t)slot[r] * a.act_s_stride;
    }
    float v[16];  // [row q][slot r] at q * kStRows + r
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
#pragma unroll 1
    for (uint32_t b0 = 0; b0 < nb; b0 += 32 * kDnJ) {
      W8 hx[kStRows][kDnJ];
      float hsc[kStRows][kDnJ];
      int sx[kStRows][kDnJ];
#pragma unroll
      for (int r = 0; r < kStRows; ++r)
#pragma unroll
        for (int j = 0; j < kDnJ; ++j) {
          const uint32_t b = b0 + lane + 32u * j;
          if (r < nr && b < nb) {
            hx[r][j] = ld_cached32(hp[r] + 32 * b);
            hsc[r][j] = __ldg(hsp[r] + b);
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) hx[r][j].v[q] = 0u;
            hsc[r][j] = 0.0f;
          }
          sx[r][j] = block_sum(hx[r][j]);
        }
#pragma unroll
      for (int q = 0; q < RW; ++q)
#pragma unroll
        for (int j = 0; j < kDnJ; ++j) {
          const uint32_t b = b0 + lane + 32u * j;
          if (b < nb) {
            const float sw = half_bits_to_float(wsc[(size_t)q * nb + b]) * scale_mul<RFMT>();
            WBlock<RFMT> wb;
            const int8_t *cp = wc + (size_t)q * rb + BB * b;
            if constexpr (RFMT == MOE_FMT_Q2S) wb.c = *(const uint2 *)cp;
            else wb.c = *(const uint4 *)cp;
            wb.prep();
#pragma unroll
            for (int r = 0; r < kStRows; ++r) {
              if (r < nr) {
                const int p = wb.dot(hx[r][j], sx[r][j]);
                v[q * kStRows + r] = __fmaf_rn((float)p, sw * hsc[r][j], v[q * kStRows + r]);
                if (TAPS && jt[q] >= 0)
                  a.tap[((size_t)slot[r] * kNTap + (size_t)jt[q]) * a.tap_nb + b] = p;
              }
            }
          }
        }
    }
    if (r0 + kStRows >= h.nrows) {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
    }
    const float tot = transpose_sum<16>(v, lane);
    const int q = lane / kStRows, r = lane % kStRows;
    if (lane < 16 && q < RW && r < nr) a.out[(size_t)slot[r] * a.out_stride + m0 + q] = tot;
  }
}

// MAT = 2: gate/up (RW = 1; routed weights of format RFMT); MAT = 1: down (RW
// rows a warp; routed weights of format RFMT, the shared expert's Q8_0)
template <int MAT, int RW, bool TAPS, int RFMT>
__global__ void __launch_bounds__(kStThreads, 1) k_stream(const StArgs a) {
  constexpr int kRows = kStGroupWarps * RW;  // rows of each matrix per stage
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(128) uint8_t ssm[];
  const uint32_t SB = a.stage_bytes;
  uint64_t *full = (uint64_t *)(ssm + (size_t)kStStages * SB);
  uint64_t *empty = full + kStStages;
  uint64_t *gbar = empty + kStStages;  // one per consumer group
  volatile int *abort_flag = (volatile int *)(gbar + kStGroups);
  float *part = (float *)(ssm + (size_t)kStStages * SB + kStBarBytes);  // gate/up half sums
  int *plan_sm = (int *)(part + kStPartFloats);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long t_entry = clock64();
  unsigned long long *tr = a.trace && blockIdx.x < kStTraceCtas
                               ? a.trace + (size_t)blockIdx.x * kStTraceStride
                               : nullptr;
  if (tid == 0) {
    for (int s = 0; s < kStStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kStGroupWarps);
    }
    for (int g = 0; g < kStGroups; ++g) mbar_init(&gbar[g], kStGroupWarps);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  PlanView P(const_cast<int *>(a.plan), a.E);
  const SmemPlan S(plan_sm, P, a.E);  // ends in a CTA barrier: the mbarriers are ready
  const int U = P.hdr[0];
  const ItemCount ic = item_count<MAT, kRows, RFMT>(a, S, U);
  const Chunks ch = chunks_of(ic);
  if (warp == kStProdWarp) {
    if (lane != 0) return;
    // activation rows the header carries: gate/up tokens (down: the slots, which
    // the consumers compute)
    constexpr int kAR = MAT == 2 ? kHdrRows : 0;
    int issued = 0, uses = 0, ends = 0;
    long long t_wait = 0;
    // g: the item being prepared, of chunk c (items up to gend)
    int c = 0, g = 0, gend = 0;
    auto advance = [&]() -> bool {
      if (g + 1 < gend) {
        ++g;
        return true;
      }
      c = (int)atomicAdd(a.queue, 1u);
      if (c >= ch.n) return false;
      g = ch.first(c);
      gend = ch.end(c);
      return true;
    };
    // the current item and its first rows' activation rows, one item ahead
    bool have = advance();
    Item cur;
    int arow[kAR + 1];
    if (have) {
      cur = item_at<MAT, kRows, RFMT>(a, S, U, ic, g);
#pragma unroll
      for (int r = 0; r < kAR; ++r)
        arow[r] = r < cur.nrows ? act_row_of<MAT>(a, cur.sh, cur.row0 + r) : 0;
    }
    int pf_row0 = -1, pf_sh = -1;
    for (int i = 0;; ++i) {
      if (*abort_flag) break;
      const int s = i % kStStages;
      const uint32_t use = (uint32_t)(i / kStStages);
      // Q8_0 down: warm this SM's L1 with the h rows of the item's first pass,
      // once per run of items with the same rows, before waiting for a stage
      // (the consumers then find them there instead of in L2).  Measured slower
      // for gate/up (x rows 3x longer) and no faster for the low-bit formats,
      // whose consumers the weight decode binds.
      if (MAT == 1 && RFMT == MOE_FMT_Q8_0 && have &&
          (cur.row0 != pf_row0 || (int)cur.sh != pf_sh)) {
        pf_row0 = cur.row0;
        pf_sh = (int)cur.sh;
        const int8_t *ab = RFMT == MOE_FMT_Q2S && !cur.sh ? a.act_t : a.act;
        const int nr = min(cur.nrows, kStRows);
        for (int r = 0; r < nr; ++r) {
          const int row = MAT == 2 ? arow[r] : cur.row0 + r;
          const char *p = (const char *)(ab + (size_t)row * a.act_stride);
          for (uint32_t off = 0; off < cur.K; off += 128)
            asm volatile("prefetch.global.L1 [%0];" ::"l"(p + off));
          const char *ps = (const char *)(a.act_s + (size_t)row * a.act_s_stride);
          for (uint32_t off = 0; off < cur.K / 8; off += 128)
            asm volatile("prefetch.global.L1 [%0];" ::"l"(ps + off));
        }
      }
      const long long tw = clock64();
      if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1u, kStWaitCycles)) {
        atomicOr(a.err, kErrTimeout);
        *abort_flag = 1;
        break;
      }
      t_wait += clock64() - tw;
      uses = i + 1;
      uint8_t *st = ssm + (size_t)s * SB;
      StageHdr *hd = (StageHdr *)st;
      if (!have) {
        // an empty header ends the loop of the group that reads item i; one for
        // each group
        hd->nrows = 0;
        mbar_arrive(&full[s]);
        if (++ends == kStGroups) break;
        continue;
      }
      if (tr && i == 0) tr[kStTrSetup] = (unsigned long long)(clock64() - t_entry);
      // the next item's lookup and permutation reads, in flight meanwhile
      const int g_cur = g;
      const bool more = advance();
      Item nxt = cur;
      int arow_n[kAR + 1];
#pragma unroll
      for (int r = 0; r < kAR; ++r) arow_n[r] = 0;
      if (more) {
        nxt = item_at<MAT, kRows, RFMT>(a, S, U, ic, g);
        const bool same = g == g_cur + 1 && nxt.row0 == cur.row0 && nxt.sh == cur.sh;
#pragma unroll
        for (int r = 0; r < kAR; ++r)
          arow_n[r] = same ? arow[r]
                           : r < nxt.nrows ? act_row_of<MAT>(a, nxt.sh, nxt.row0 + r) : 0;
      }
      // header, then the weight copies
      hd->row0 = cur.row0;
      hd->nrows = cur.nrows;
      hd->n0 = cur.n0;
      hd->sh = cur.sh ? 1 : 0;
      hd->K = (int)cur.K;
#pragma unroll
      for (int r = 0; r < kAR; ++r) hd->act_row[r] = arow[r];
      const uint32_t qb = (uint32_t)cur.nf * cur.rb, sb = (uint32_t)cur.nf * (cur.K / 16);
      uint8_t *w = st + kStHdrBytes;
      mbar_expect_tx(&full[s], MAT * (qb + sb));
#pragma unroll
      for (int m = 0; m < MAT; ++m) {
        bulk_g2s(w + (size_t)m * qb, cur.q[m], qb, &full[s]);
        bulk_g2s(w + (size_t)MAT * qb + (size_t)m * sb, cur.s[m], sb, &full[s]);
      }
      ++issued;
      have = more;
      cur = nxt;
#pragma unroll
      for (int r = 0; r < kAR; ++r) arow[r] = arow_n[r];
    }
    // no copy may still be landing when the CTA exits: wait (bounded) for the
    // last use of each stage (at once in a normal run: consumed or an empty
    // header)
    for (int i = max(0, uses - kStStages); i < uses; ++i)
      if (!mbar_wait(&full[i % kStStages], (uint32_t)(i / kStStages) & 1u, kStWaitCycles))
        atomicOr(a.err, kErrTimeout);
    // the last producer out zeroes the queue for the next call (every other
    // producer has taken its last chunk before it counts itself out)
    __threadfence();
    if (atomicAdd(a.queue + 1, 1u) == gridDim.x - 1) {
      atomicExch(a.queue, 0u);
      atomicExch(a.queue + 1, 0u);
    }
    if (tr) {
      tr[kStTrProdWait] = (unsigned long long)t_wait;
      tr[kStTrItems] = (unsigned long long)issued;
      tr[kStTrProdTotal] = (unsigned long long)(clock64() - t_entry);
    }
    return;
  }
  const int gi = warp / kStGroupWarps, wi = warp % kStGroupWarps;
  uint32_t par = 0;  // gate/up: pass parity (partial-sum buffer, group barrier phase)
  long long c_wait = 0, c_work = 0;
  for (int i = gi; !*abort_flag; i += kStGroups) {
    const int s = i % kStStages;
    const uint32_t use = (uint32_t)(i / kStStages);
    const long long tw = clock64();
    // item i - 4 released (one phase behind at most), then item i's bytes
    if ((use > 0 && !mbar_wait(&empty[s], (use - 1) & 1u, kStWaitCycles)) ||
        !mbar_wait(&full[s], use & 1u, kStWaitCycles)) {
      atomicOr(a.err, kErrTimeout);
      *abort_flag = 1;
      break;
    }
    const long long tg = clock64();
    c_wait += tg - tw;
    const uint8_t *st = ssm + (size_t)s * SB;
    // the header's scalars in registers; gate/up reads its token list in place
    const StageHdr *hp = (const StageHdr *)st;
    if (hp->nrows == 0) break;  // no more items for this group
    StageHdr h;
    h.row0 = hp->row0;
    h.nrows = hp->nrows;
    h.n0 = hp->n0;
    h.sh = hp->sh;
    h.K = hp->K;
    if (MAT == 2) {
      float *gpart = part + (size_t)gi * kStPartPerGroup;
      bool ok;
      if constexpr (RFMT != MOE_FMT_Q8_0) {
        ok = !h.sh ? gateup_stage_lb<RFMT, TAPS>(a, h, hp->act_row, st + kStHdrBytes, wi, lane,
                                                 gpart, &gbar[gi], par, &empty[s])
                   : gateup_stage<TAPS>(a, h, hp->act_row, st + kStHdrBytes, wi, lane, gpart,
                                        &gbar[gi], par, &empty[s]);
      } else {
        ok = gateup_stage<TAPS>(a, h, hp->act_row, st + kStHdrBytes, wi, lane, gpart, &gbar[gi],
                                par, &empty[s]);
      }
      if (!ok) {
        atomicOr(a.err, kErrTimeout);
        *abort_flag = 1;
        break;
      }
    } else {
      if constexpr (RFMT != MOE_FMT_Q8_0) {
        if (!h.sh) down_stage_lb<RFMT, RW, TAPS>(a, h, st + kStHdrBytes, wi, lane, &empty[s]);
        else down_stage<RW, TAPS>(a, h, st + kStHdrBytes, wi, lane, &empty[s]);
      } else {
        down_stage<RW, TAPS>(a, h, st + kStHdrBytes, wi, lane, &empty[s]);
      }
    }
    c_work += clock64() - tg;
  }
  if (tr && lane == 0) {
    tr[kStTrConsWait + warp] = (unsigned long long)c_wait;
    tr[kStTrConsWork + warp] = (unsigned long long)c_work;
  }
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

size_t stream_smem(uint32_t stage_bytes, uint32_t E) {
  return (size_t)kStStages * stage_bytes + kStBarBytes + 4 * kStPartFloats + smem_plan_bytes(E);
}

// bytes of a stage: header, MAT matrices of `rows` weight rows of K weights in
// format fmt and K/32 fp16 scales
uint64_t stage_bytes_for(int mat, uint32_t rows, uint32_t K, int fmt = MOE_FMT_Q8_0) {
  return kStHdrBytes + (uint64_t)mat * rows * (row_bytes(fmt, K) + K / 16);
}

// a gate/up stage holds a routed item or a shared-expert item (4 Q8_0 features)
uint64_t gateup_stage_bytes(const moe_desc &D) {
  const int fmt = D.routed_fmt;
  const uint32_t fpi = fmt == MOE_FMT_Q2S    ? fpi_of<MOE_FMT_Q2S>()
                       : fmt == MOE_FMT_E2M1 ? fpi_of<MOE_FMT_E2M1>()
                                             : fpi_of<MOE_FMT_Q8_0>();
  uint64_t b = stage_bytes_for(2, fpi, D.d, fmt);
  if (D.f_shared) b = std::max<uint64_t>(b, stage_bytes_for(2, kStGroupWarps, D.d));
  return b;
}

// down rows a warp takes per stage: Q8_0 routed weights the most of 6, 4, 2, 1,
// low-bit ones (whose rows are small) of 8, 4, whose stage fits (routed rows and
// the shared expert's Q8_0 rows), whose items tile d and whose copies are whole
// 16-byte units
int down_rw(const moe_desc &D) {
  const bool low = D.routed_fmt != MOE_FMT_Q8_0;
  if (row_bytes(D.routed_fmt, D.f) % 16) return 0;
  for (int rw : {8, 6, 4, 2, 1}) {
    if (low ? (rw != 8 && rw != 4) : rw == 8) continue;
    const uint32_t rows = (uint32_t)kStGroupWarps * rw;
    if (D.d % rows) continue;
    if (stage_bytes_for(1, rows, D.f, D.routed_fmt) > kStStageMax) continue;
    if (D.f_shared && stage_bytes_for(1, rows, D.f_shared) > kStStageMax) continue;
    if ((rw * D.f / 4) % 16 || (rw * D.f_shared / 4) % 16) continue;
    if ((rows * row_bytes(D.routed_fmt, D.f)) % 16) continue;
    return rw;
  }
  return 0;
}

template <int MAT, int RW, bool TAPS, int RFMT = MOE_FMT_Q8_0>
cudaError_t run_stream(const Ctx &c, const StArgs &a) {
  static bool big_smem = false;
  auto kern = k_stream<MAT, RW, TAPS, RFMT>;
  const size_t smem = stream_smem(a.stage_bytes, c.desc.n_expert);
  if (!big_smem) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStSmemMax);
    if (e != cudaSuccess) return e;
    big_smem = true;
  }
  const cudaError_t e = launch_k(kern, c.sm_count, kStThreads, smem, c.stream, c.chained, a);
  c.chained = true;
  return e;
}

}  // namespace

// gate/up on the streamed GEMV (any routed format): d a multiple of 128 (a
// 4-feature scale slice is a whole number of 16-byte copies; K halves of whole
// blocks) and at most 6144 (3 blocks a lane and row); 16-byte aligned scale
// planes
bool stream_gateup_ok(const Ctx &c) {
  const moe_desc &D = c.desc;
  const uint32_t jmax = D.routed_fmt == MOE_FMT_Q8_0 ? kGuJ : kGuJLowBit;
  if (D.d % 128 || D.d > 64u * 32u * jmax) return false;
  if (gateup_stage_bytes(D) > kStStageMax) return false;
  if (!aligned16(c.wts.gate.scale) || !aligned16(c.wts.up.scale)) return false;
  if (D.f_shared && (!aligned16(c.wts.s_gate.scale) || !aligned16(c.wts.s_up.scale))) return false;
  // bulk copies start on 16-byte boundaries (2-bit planes need only 8)
  if (!aligned16(c.wts.gate.q) || !aligned16(c.wts.up.q)) return false;
  if (D.f_shared && (!aligned16(c.wts.s_gate.q) || !aligned16(c.wts.s_up.q))) return false;
  return true;
}

// down (any routed format): an item shape that tiles d with 16-byte copies
// (codes and RW * K / 4 bytes of scales a stage and a row offset); 16-byte
// aligned scale planes
bool stream_down_ok(const Ctx &c) {
  const moe_desc &D = c.desc;
  if (down_rw(D) == 0) return false;
  // 2-bit routed weights read the transposed h codes
  if (D.routed_fmt == MOE_FMT_Q2S && !c.L.ht) return false;
  if (!aligned16(c.wts.down.scale) || !aligned16(c.wts.down.q)) return false;
  if (D.f_shared && (!aligned16(c.wts.s_down.scale) || !aligned16(c.wts.s_down.q)))
    return false;
  return true;
}

cudaError_t launch_gateup_stream(const Ctx &c, const int32_t *perm) {
  const moe_desc &D = c.desc;
  StArgs a;
  memset(&a, 0, sizeof a);
  a.plan = (const int *)(c.ws + c.L.plan);
  a.E = D.n_expert;
  a.k = D.top_k;
  a.d = D.d;
  a.f = D.f;
  a.fs = D.f_shared;
  a.R = c.R;
  a.K = a.Ks = D.d;
  a.q[0] = (const int8_t *)c.wts.gate.q;
  a.q[1] = (const int8_t *)c.wts.up.q;
  a.sc[0] = c.wts.gate.scale;
  a.sc[1] = c.wts.up.scale;
  a.sq[0] = (const int8_t *)c.wts.s_gate.q;
  a.sq[1] = (const int8_t *)c.wts.s_up.q;
  a.ssc[0] = c.wts.s_gate.scale;
  a.ssc[1] = c.wts.s_up.scale;
  a.rows_per_slot = D.f;
  a.eslot = c.wts.expert_slot;
  a.act = (const int8_t *)(c.ws + c.L.xq);
  a.act_t = c.L.xt ? (const int8_t *)(c.ws + c.L.xt) : nullptr;
  a.act_s = (const float *)(c.ws + c.L.xs);
  a.act_stride = D.d;
  a.act_s_stride = D.d / 32;
  a.perm = perm;
  a.out = (float *)(c.ws + c.L.h);
  a.out_stride = c.fmax;
  const bool taps = (D.flags & MOE_FLAG_DEBUG_TAPS) != 0;
  a.tap = taps ? (int32_t *)(c.ws + c.L.tap_gu) : nullptr;
  a.tap_nb = D.d / 32;
  a.err = (uint32_t *)(c.ws + c.L.err);
  a.stage_bytes = (uint32_t)gateup_stage_bytes(D);
  a.queue = (uint32_t *)(c.ws + c.L.sync) + kQueueStreamGateup;
  a.trace = (D.flags & MOE_FLAG_TRACE) && c.L.trace
                ? (unsigned long long *)(c.ws + c.L.trace) + kStTraceBase
                : nullptr;
  switch (D.routed_fmt) {
    case MOE_FMT_Q2S:
      return taps ? run_stream<2, 1, true, MOE_FMT_Q2S>(c, a)
                  : run_stream<2, 1, false, MOE_FMT_Q2S>(c, a);
    case MOE_FMT_E2M1:
      return taps ? run_stream<2, 1, true, MOE_FMT_E2M1>(c, a)
                  : run_stream<2, 1, false, MOE_FMT_E2M1>(c, a);
    default: return taps ? run_stream<2, 1, true>(c, a) : run_stream<2, 1, false>(c, a);
  }
}

cudaError_t launch_down_stream(const Ctx &c) {
  const moe_desc &D = c.desc;
  const int rw = down_rw(D);
  StArgs a;
  memset(&a, 0, sizeof a);
  a.plan = (const int *)(c.ws + c.L.plan);
  a.E = D.n_expert;
  a.k = D.top_k;
  a.d = D.d;
  a.f = D.f;
  a.fs = D.f_shared;
  a.R = c.R;
  a.K = D.f;
  a.Ks = D.f_shared;
  a.out_per_e = D.d;
  a.q[0] = (const int8_t *)c.wts.down.q;
  a.sc[0] = c.wts.down.scale;
  a.sq[0] = (const int8_t *)c.wts.s_down.q;
  a.ssc[0] = c.wts.s_down.scale;
  a.rows_per_slot = D.d;
  a.eslot = c.wts.expert_slot;
  a.act = (const int8_t *)(c.ws + c.L.hq);
  a.act_t = c.L.ht ? (const int8_t *)(c.ws + c.L.ht) : nullptr;
  a.act_s = (const float *)(c.ws + c.L.hs);
  a.act_stride = c.fmax;
  a.act_s_stride = c.fmax / 32;
  a.out = (float *)(c.ws + c.L.o);
  a.out_stride = D.d;
  const bool taps = (D.flags & MOE_FLAG_DEBUG_TAPS) != 0;
  a.tap = taps ? (int32_t *)(c.ws + c.L.tap_dn) : nullptr;
  a.tap_nb = c.fmax / 32;
  a.err = (uint32_t *)(c.ws + c.L.err);
  const uint32_t rows = (uint32_t)kStGroupWarps * rw;
  a.stage_bytes = (uint32_t)std::max<uint64_t>(stage_bytes_for(1, rows, D.f, D.routed_fmt),
                                                D.f_shared ? stage_bytes_for(1, rows, D.f_shared)
                                                           : 0);
  a.queue = (uint32_t *)(c.ws + c.L.sync) + kQueueStreamDown;
  a.trace = (D.flags & MOE_FLAG_TRACE) && c.L.trace
                ? (unsigned long long *)(c.ws + c.L.trace) + kStTraceBase + kStTraceDown
                : nullptr;
  if (D.routed_fmt == MOE_FMT_Q2S || D.routed_fmt == MOE_FMT_E2M1) {
    // low-bit routed rows: 8 rows a warp where the layer allows it (the
    // 192-expert layers), else the Q8_0 kernel's choices
    const bool q2 = D.routed_fmt == MOE_FMT_Q2S;
    switch (rw) {
      case 8:
        return q2 ? (taps ? run_stream<1, 8, true, MOE_FMT_Q2S>(c, a)
                          : run_stream<1, 8, false, MOE_FMT_Q2S>(c, a))
                  : (taps ? run_stream<1, 8, true, MOE_FMT_E2M1>(c, a)
                          : run_stream<1, 8, false, MOE_FMT_E2M1>(c, a));
      case 4:
        return q2 ? (taps ? run_stream<1, 4, true, MOE_FMT_Q2S>(c, a)
                          : run_stream<1, 4, false, MOE_FMT_Q2S>(c, a))
                  : (taps ? run_stream<1, 4, true, MOE_FMT_E2M1>(c, a)
                          : run_stream<1, 4, false, MOE_FMT_E2M1>(c, a));
      default:
        return cudaErrorInvalidValue;  // down_rw gives low-bit layers 8 or 4 (or 0)
    }
  }
  switch (rw) {
    case 6: return taps ? run_stream<1, 6, true>(c, a) : run_stream<1, 6, false>(c, a);
    case 4: return taps ? run_stream<1, 4, true>(c, a) : run_stream<1, 4, false>(c, a);
    case 2: return taps ? run_stream<1, 2, true>(c, a) : run_stream<1, 2, false>(c, a);
    default: return taps ? run_stream<1, 1, true>(c, a) : run_stream<1, 1, false>(c, a);
  }
}

}  // namespace moe
