// decode_fused.cu -- the whole layer for one or two tokens in one persistent kernel.
//
// Single-token decode moves ~361 MB of expert weights (8 routed experts + the
// shared expert of a GLM-5.2-sized layer) and almost no arithmetic, so the
// layer is bound by HBM bandwidth and by anything that leaves HBM idle:
// launch gaps between small kernels, the router's latency, and the drain/ramp
// between the gate/up and the down projection.  This kernel removes all three.
//
//  * One CTA per SM (cooperative launch, all CTAs co-resident), 16 consumer
//    warps and 1 producer warp.  The producer lane streams weight rows with
//    cp.async.bulk (the bulk-copy/TMA engine, one-CTA copies, no multicast) into
//    a ring of up to 8 shared-memory stages guarded by mbarriers; consumers
//    compute from shared memory with dp4a.
//  * Every CTA routes the tokens itself (sigmoid + bias, top-k in registers,
//    stable permutation) from the same inputs, so no CTA waits on another for
//    the routing; CTA 0 also writes the routing arrays to the workspace.  While
//    the consumers route, the producer is already streaming the shared expert,
//    whose items need no routing.
//  * Work comes from one global queue, handed out in this order: gate/up items
//    of the shared expert (known before the routing), gate/up items of the
//    routed experts, then down items of every expert.  A gate/up item is 32 features of one expert (one int8
//    block of h, requantised by the CTA that computed it) in stages of 8
//    features; a down item is a chunk of output rows of one expert.
//  * A down item needs its expert's h complete: the producer waits on a
//    per-expert counter (after issuing the stage's weight copies) before it
//    copies the h codes in.  Because every gate/up item is handed out before
//    any down item and all CTAs are resident, every such wait ends.
//  * The combine (y = o_shared + sum_j w_j o_j, fixed order) runs at the end,
//    after a grid barrier on the expert outputs o, split over all threads.
//  * Every wait is bounded; on timeout the kernel flags kErrTimeout and exits.
// Per-expert batches of the selected experts only, read once per call: the
// indexed per-expert FFN of NeutronStar README, "MTP speculative decoding".
#include "stream_ptx.cuh"

namespace moe {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kProducerWarp = kConsumerWarps;       // lane 0 issues the weight copies
constexpr int kPublisherWarp = kConsumerWarps + 1;  // lane 0 does the gpu-scope atomics
constexpr int kThreads = (kConsumerWarps + 2) * 32;
constexpr int kPubCap = 64;      // events in flight from the CTA's warps to its publisher
constexpr int kRouteWarp0 = 1;   // first routing warp (not on the producer's SM sub-partition)
constexpr int kMaxT = 2;
constexpr int kMaxR = 64;        // routed rows (T * top_k)
constexpr int kBFeat = 8;        // features per gate/up stage
constexpr int kKSplit = kConsumerWarps / kBFeat;  // K parts per feature (one warp each)
constexpr int kBItemFeat = 32;   // features per gate/up item: one quantisation block
constexpr int kDnRows = kBFeat == 8 ? 3 : 2;  // down rows per warp and pass (~43 / ~21 a stage)
constexpr int kXRegs = kBFeat == 8 ? 6 : 4;   // x chunks per lane in registers (d <= 6144 / 8192)
constexpr int kMaxStages = 8;
// x quads (128 floats) a quantising warp takes at T tokens: d <= 16*kKSplit*32*kXRegs
// = 6144 gives 48 quads per token, over 15 warps at T=1 and 14 at T=2
constexpr int kMaxQuadsPerToken = 16 * kKSplit * 32 * kXRegs / 128;
template <int NT>
__host__ __device__ constexpr int x_quads() {
  return (NT * kMaxQuadsPerToken + kConsumerWarps - NT - 1) / (kConsumerWarps - NT);
}
// partial-sum buffers of gate/up items.  The warp that requantises item i reads
// buffer i % kPartBufs after releasing the item's last stage; the other warps
// can then run at most kMaxStages stages ahead, i.e. into item i + 2 at most
// (items are 4 stages), so three buffers keep its buffer from being refilled.
constexpr int kPartBufs = 3;
static_assert(kMaxStages <= (kPartBufs - 1) * (kBItemFeat / kBFeat),
              "the stage ring could let a warp reach an item whose buffer is still read");
constexpr uint32_t kSyncInts = MOE_SYNC_BYTES / 4;
constexpr long long kWaitCycles = 4000000000ll;     // ~2 s at 2 GHz: a wait gives up after this
constexpr long long kStallTestCycles = 20000000ll;  // ~10 ms under MOE_FLAG_TEST_STALL

enum : int { kKindB = 0, kKindC = 1, kKindEnd = 2 };

// MOE_FLAG_TRACE words per CTA (absolute times in ns of %globaltimer, durations
// in SM clock cycles)
enum : int {
  kTrStart = 0,        // kernel entry (ns)
  kTrXqDone = 1,       // x quantised (ns)
  kTrFirstStage = 2,   // first stage ready for the consumers (ns)
  kTrWaitFull = 3,     // consumers waiting for stage data (cycles)
  kTrWaitReady = 4,    // consumers waiting for an expert's h (cycles)
  kTrStagesB = 5,      // gate/up stages consumed
  kTrStagesC = 6,      // down stages consumed
  kTrConsEnd = 7,      // consumers leave (ns)
  kTrWaitEmpty = 8,    // producer waiting for a free stage (cycles)
  kTrWaitRoute = 9,    // producer waiting for the routing result (cycles)
  kTrItems = 10,       // items taken by this CTA
  kTrComputeB = 11,    // consumer cycles in gate/up stages
  kTrComputeC = 12,    // consumer cycles in down stages
  kTrCombine = 13,     // cycles in the final combine
  kTrRouteDone = 14,   // routing known to the producer (ns)
  kTrProdEnd = 15,     // producer leaves (ns)
  kTrRouteLoaded = 16, // selection scores computed (ns)
  kTrRouteTopk = 17,   // publisher: cycles in its gpu-scope atomics
  kTrRoutePerm = 18,   // permutation and active list done (ns)
  kTrExit = 19,        // CTA leaves the kernel (ns)
  kTrW5WaitFull = 20,  // consumer warp 5 (no requant duty): waiting for stage data (cycles)
  kTrW5ComputeB = 21,  // consumer warp 5: cycles in gate/up stages
  kTrW5ComputeC = 22,  // consumer warp 5: cycles in down stages
  kTrItemEnd = 23,     // consumer warp 0: cycles at item ends (barrier + requant)
  // 24..26: routing warp 0 after its top-k, weights and permutation (ns);
  // 27: the CTA's router partial sums written (ns)
  kTrLatIssueGot = 28, // producer, over reused slots: cycles from issuing a stage to
  kTrLatGotRel = 29,   //   consumer warp 0 having its data, from then to warp 0's
  kTrLatRelEmpty = 30, //   release, and from that to the producer seeing the slot
  kTrLatSamples = 31,  //   empty; and the number of such stages
  kTraceWords = 32
};

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct StageDesc {
  int kind;
  int e;           // expert id, E = shared expert
  int we;          // routed: the expert's weight slot
  int first;       // B: first feature of the stage; C: first output row
  int count;       // B: features (8); C: output rows
  int sub;         // B: sub-stage in the item (0..3)
  int item_first;  // B: first feature of the item; C: chunk index
  int nrows;       // token rows of this expert
  int slot[kMaxT];
  int tok[kMaxT];
};

struct FusedArgs {
  uint32_t E, k, d, f, fs, T, R, fmax;
  // the routed experts this call computes, [e_lo, e_hi), and the shared
  // expert's width if the call adds it, else 0 (an expert-parallel rank's share)
  uint32_t e_lo, e_hi, fs_on;
  float s;
  uint32_t score;  // moe_score
  const float *x, *logits, *bias;
  // router logits computed in the kernel (wr non-null): W_router [E][d] fp32, the
  // segment partial sums rseg [T][E][nseg] (workspace), logits_out [T][E]
  const float *wr;
  float *rseg, *logits_out;
  uint32_t nseg;
  const int8_t *gq, *uq, *dq, *sgq, *suq, *sdq;
  const uint16_t *gs, *us, *ds, *sgs, *sus, *sds;
  const int32_t *eslot;  // expert -> weight slot (moe_weights.expert_slot), or null
  uint32_t n_slots;      // slots in the routed weight planes
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
  // MOE_FLAG_DEBUG_TAPS: the int32 block dots of the tapped features and outputs
  // (moe.h tap layout: tap_gu[slot][2][kNTap][d/32], tap_dn[slot][kNTap][fmax/32])
  int32_t *tap_gu, *tap_dn;
  uint32_t *sync;  // see SyncView
  uint32_t *err;
  uint32_t c_rows, n_chunks, n_stages, stage_bytes;
  uint32_t part_bytes;    // the part[] region, which also holds the routing scores
  long long wait_cycles;  // budget of every bounded wait
  unsigned long long *trace;  // MOE_FLAG_TRACE: kTraceWords per CTA, else null
  int stall_test;         // MOE_FLAG_TEST_STALL: never publish the routing result
};

// Counters at a fixed workspace offset (moe.h: MOE_SYNC_BYTES from offset 256).
// They are zero before a call and the last CTA to finish zeroes them again, so
// no per-call memset is needed (a workspace must be zero-filled once after it
// is allocated).  diag[] keeps the first timeout's site for the host.
struct SyncView {
  uint32_t *queue, *diag, *ready, *fin, *gen;
  uint32_t n_clear;  // words from queue through ready[] (diag words are kept)
  __device__ SyncView(uint32_t *base, uint32_t E) {
    queue = base;      // [0]; [1]: CTAs whose router partial sums are written
    diag = base + 2;   // [2], [3]
    ready = base + 4;  // [E+1] gate/up items finished per expert
    // the two counters that carry over between calls sit at the end of the area,
    // clear of ready[] for any E, so calls of different E may share a workspace
    fin = base + kSyncInts - 2;  // CTAs whose expert outputs o are written, counting up
    gen = base + kSyncInts - 1;  // calls completed: this call's fin target is (gen+1)*grid
    n_clear = 4 + E + 1;
  }
};

// CTA-local control words and the publisher's event ring.  An event: expert e's
// h rows of one gate/up item are written.
struct SharedCtl {
  int abort;          // a wait gave up: stop issuing, skip the combine
  uint32_t gen;       // SyncView::gen at the call's start
  int writers_done;   // consumer warps + producer that will post no more events
  int item_cnt[kPartBufs];  // consumer warps done with an item, by b_items % kPartBufs
  int pub_head;       // events reserved
  int pub_tail;       // events taken by the publisher
  int pub_ev[kPubCap];
  int pub_seq[kPubCap];  // event i is valid when pub_seq[i % kPubCap] == i + 1
  long long t_issue[kMaxStages], t_got[kMaxStages], t_rel[kMaxStages];  // MOE_FLAG_TRACE
};

// Routing of the call, held in shared memory by every CTA.
struct RouteSmem {
  int idx[kMaxR];     // expert of row r = t*k + j
  float w[kMaxR];     // its combine weight
  int pos[kMaxR];     // slot of row r (stable sort by expert)
  int tok[kMaxR];     // token of slot p
  int act_e[kMaxR];   // active routed experts in id order, their weight slot, first row slot and rows
  int act_w[kMaxR];
  int act_row0[kMaxR];
  int act_rows[kMaxR];
  int row_at[kMaxR];  // row at slot p
  uint32_t first_bits[2];  // slot p opens an expert's run (bit p)
  int U;              // active routed experts
  int bad_slot;       // an active expert's weight slot is outside [0, n_slots)
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}


// one thread publishes the CTA's prior writes (made visible to it by a CTA
// barrier) with a gpu-scope release reduction
__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}


// a bounded wait gave up: flag the error word (kErrTimeout plus the wait site in
// bits 8..15) and keep the first site / CTA / detail in sync[2], sync[3]
__device__ __noinline__ void report_timeout(const FusedArgs &a, uint32_t site, uint32_t detail) {
  atomicOr(a.err, kErrTimeout | (1u << (8 + site)));
  if (atomicCAS(&a.sync[2], 0u, (site << 24) | (blockIdx.x & 0xFFFFFFu)) == 0u)
    a.sync[3] = detail;
}

// hand an event to the CTA's publisher warp (any thread; bounded wait for room)
__device__ __noinline__ void pub_post(const FusedArgs &a, SharedCtl &ctl, int ev) {
  const int i = atomicAdd(&ctl.pub_head, 1);
  const long long t0 = clock64();
  while (i - *(volatile int *)&ctl.pub_tail >= kPubCap) {
    if (clock64() - t0 > a.wait_cycles) {
      report_timeout(a, 5, (uint32_t)i);
      *(volatile int *)&ctl.abort = 1;
      return;
    }
  }
  ctl.pub_ev[i % kPubCap] = ev;
  __threadfence_block();
  *(volatile int *)&ctl.pub_seq[i % kPubCap] = i + 1;
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}


__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------- routing (every CTA)
// Every CTA routes the tokens itself from the same inputs, so all CTAs hold the
// same routing in shared memory without waiting on one another; CTA 0 also
// writes idx, w, off, perm, pos and the plan's active list to the workspace.
// This code runs once per call with a cold instruction cache (each new line of
// code costs a round trip to L2 or HBM), so it is kept compact -- rolled loops,
// no unrolled sorting network -- and only the T routing warps run it, while the
// other consumer warps quantise x.

__device__ __forceinline__ void route_bar_sync(uint32_t T) {
  asm volatile("bar.sync 3, %0;" ::"r"(T * 32) : "memory");
}

// scores p(l) (sigmoid or sqrt-softplus of the logit) and selection scores
// c = p + bias of all T*E (token, expert) pairs, into sg and sc (every consumer
// thread; a consumer barrier follows).  With the router in the kernel, the
// logit is the sum of its segment partials in ascending order, read through L2
// (other CTAs wrote them), and CTA 0 stores it for the caller.
constexpr uint32_t kMaxSeg = 8;  // router segments: d <= 8192
__device__ void route_scores(const FusedArgs &a, float *sc, float *sg, float pre_l, float pre_b) {
#pragma unroll 1
  for (uint32_t i = threadIdx.x; i < a.T * a.E; i += kConsumerWarps * 32) {
    const bool first = i == threadIdx.x;  // its logit (if given) and bias came at entry
    float l;
    if (a.wr) {
      const float *ps = a.rseg + (size_t)i * a.nseg;
      float v[kMaxSeg];
#pragma unroll
      for (uint32_t g = 0; g < kMaxSeg; ++g) v[g] = g < a.nseg ? __ldcg(ps + g) : 0.0f;
      l = v[0];
#pragma unroll
      for (uint32_t g = 1; g < kMaxSeg; ++g)
        if (g < a.nseg) l = __fadd_rn(l, v[g]);
      if (blockIdx.x == 0) a.logits_out[i] = l;
    } else {
      l = first ? pre_l : __ldg(a.logits + i);
    }
    const float p = score_rn(l, a.score);
    sg[i] = p;
    sc[i] = __fadd_rn(p, first ? pre_b : __ldg(a.bias + i % a.E));
  }
}

// order-preserving unsigned key of a selection score (scores are never NaN; -0
// takes +0's key).  Key 0 is below every score's key: it marks an absent or
// already selected entry.
__device__ __forceinline__ uint32_t score_key(float c) {
  uint32_t b = __float_as_uint(c);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// top-k of one token by one warp, E <= 32*NV: lane l holds the keys of experts
// l + 32i (ct: the token's selection scores).  Each round takes the lane's
// best key (strict '>' over ascending i keeps the lower expert), the warp's
// largest key (redux) and the lowest expert holding it (redux), and the
// winning lane retires that entry.
template <int NV>
__device__ __forceinline__ void topk_regs(const float *ct, uint32_t E, uint32_t k, int lane,
                                          int *out) {
  uint32_t v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const uint32_t e = (uint32_t)lane + 32u * i;
    v[i] = e < E ? score_key(ct[e]) : 0u;
  }
#pragma unroll 1
  for (uint32_t j = 0; j < k; ++j) {
    uint32_t bk = v[0];
    int bi = 0;
#pragma unroll
    for (int i = 1; i < NV; ++i)
      if (v[i] > bk) {
        bk = v[i];
        bi = i;
      }
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t be =
        __reduce_min_sync(0xffffffffu, bk == m ? (uint32_t)lane + 32u * bi : 0xffffffffu);
    if ((int)(be & 31u) == lane) {
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (i == (int)(be >> 5)) v[i] = 0u;
    }
    if (lane == 0) out[j] = (int)be;
  }
}

// the same selection for E > 512: the keys replace the selection scores in
// shared memory, and each round scans them with a stride of 32
__device__ __noinline__ void topk_scan(float *ct, uint32_t E, uint32_t k, int lane, int *out) {
  uint32_t *kt = reinterpret_cast<uint32_t *>(ct);
#pragma unroll 1
  for (uint32_t e = lane; e < E; e += 32) kt[e] = score_key(ct[e]);
#pragma unroll 1
  for (uint32_t j = 0; j < k; ++j) {
    uint32_t bk = 0u, be_l = 0xffffffffu;
#pragma unroll 1
    for (uint32_t e = lane; e < E; e += 32) {
      const uint32_t v = kt[e];
      if (v > bk) {
        bk = v;
        be_l = e;
      }
    }
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t be = __reduce_min_sync(0xffffffffu, bk == m ? be_l : 0xffffffffu);
    if ((int)(be & 31u) == lane) kt[be] = 0u;
    if (lane == 0) out[j] = (int)be;
  }
}

// warps 0..T-1: warp t selects token t's top_k (keys in registers for E <= 512,
// else k rounds of a strided scan of the scores); then the stable permutation
// (rows by expert, then row order) and the active list, with the T warps'
// threads as the R <= 64 rows.  route_scores has filled sc and sg.
__device__ void route_select(const FusedArgs &a, RouteSmem &rs, float *sc, const float *sg,
                             unsigned long long *tr) {
  const int tid = (int)threadIdx.x - kRouteWarp0 * 32, lane = tid & 31, t = tid >> 5;
  const uint32_t E = a.E, k = a.k, T = a.T;
  const int R = (int)a.R;
  float *ct = sc + (size_t)t * E;
  const float *gt = sg + (size_t)t * E;
  if (tid == 0) rs.bad_slot = 0;  // read after the barriers below
  if (E <= 256) {
    topk_regs<8>(ct, E, k, lane, rs.idx + t * k);
  } else if (E <= 512) {
    topk_regs<16>(ct, E, k, lane, rs.idx + t * k);
  } else {
    topk_scan(ct, E, k, lane, rs.idx + t * k);
  }
  __syncwarp();
  if (tr && tid == 0) tr[24] = global_ns();
  // lane j < k: the score of slot j; w = s * p_j / sum_j p_j (in order)
  const float my_sigma = (uint32_t)lane < k ? gt[rs.idx[t * k + lane]] : 0.0f;
  float sum = 0.0f;
#pragma unroll 1
  for (uint32_t j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, my_sigma, j));
  if ((uint32_t)lane < k) rs.w[t * k + lane] = __fmul_rn(a.s, __fdiv_rn(my_sigma, sum));
  if (tr && tid == 0) tr[25] = global_ns();
  route_bar_sync(T);
  // slot of row r = rows before it in (expert, row) order
  if (tid < R) {
    const int e = rs.idx[tid];
    int rank = 0;
#pragma unroll 1
    for (int r = 0; r < R; ++r) {
      const int er = rs.idx[r];
      rank += (er < e || (er == e && r < tid)) ? 1 : 0;
    }
    rs.pos[tid] = rank;
    rs.row_at[rank] = tid;
    rs.tok[rank] = tid / (int)k;
    if (blockIdx.x == 0) {
      a.idx[tid] = e;
      a.w[tid] = rs.w[tid];
      a.pos[tid] = rank;
      a.perm[rank] = tid;
    }
  }
  if (blockIdx.x == 0) {
#pragma unroll 1
    for (uint32_t e = tid; e <= E; e += T * 32) {
      int c = 0;
#pragma unroll 1
      for (int r = 0; r < R; ++r) c += rs.idx[r] < (int)e ? 1 : 0;
      a.off[e] = c;
    }
  }
  if (tr && tid == 0) tr[26] = global_ns();
  route_bar_sync(T);
  // active list: slot p opens an entry when its expert differs from slot p-1's;
  // the entry's index is the number of openings before p
  {
    const int p = tid;
    const int e = p < R ? rs.idx[rs.row_at[p]] : -1;
    const bool first = p < R && (p == 0 || rs.idx[rs.row_at[p - 1]] != e);
    const uint32_t bits = __ballot_sync(0xffffffffu, first);
    if (lane == 0) rs.first_bits[t] = bits;
    if (T == 1 && tid == 0) rs.first_bits[1] = 0u;
  }
  route_bar_sync(T);
  if (tid < R) {
    const int p = tid;
    const int e = rs.idx[rs.row_at[p]];
    const uint32_t b0 = rs.first_bits[0], b1 = rs.first_bits[1];
    if (((p < 32 ? b0 : b1) >> (p & 31)) & 1u) {
      const int u = p < 32 ? __popc(b0 & ((1u << p) - 1u))
                           : __popc(b0) + __popc(b1 & ((1u << (p - 32)) - 1u));
      int rows = 1;
#pragma unroll 1
      for (int q = p + 1; q < R && rs.idx[rs.row_at[q]] == e; ++q) ++rows;
      rs.act_e[u] = e;
      rs.act_row0[u] = p;
      rs.act_rows[u] = rows;
      rs.act_w[u] = a.eslot ? __ldg(a.eslot + e) : e;
    }
  }
  route_bar_sync(T);
  if (tid == 0) {
    // keep the experts this call computes, in order; only their weight slots
    // must be valid
    const int U = __popc(rs.first_bits[0]) + __popc(rs.first_bits[1]);
    int V = 0;
#pragma unroll 1
    for (int u = 0; u < U; ++u) {
      const int e = rs.act_e[u];
      if ((uint32_t)e < a.e_lo || (uint32_t)e >= a.e_hi) continue;
      rs.act_e[V] = e;
      rs.act_w[V] = rs.act_w[u];
      rs.act_row0[V] = rs.act_row0[u];
      rs.act_rows[V] = rs.act_rows[u];
      if ((uint32_t)rs.act_w[V] >= a.n_slots) rs.bad_slot = 1;
      if (blockIdx.x == 0) {
        PlanView P(a.plan, E);
        P.act_e[V] = e;
        P.act_row0[V] = rs.act_row0[V];
        P.act_rows[V] = rs.act_rows[V];
      }
      ++V;
    }
    rs.U = V;
    if (rs.bad_slot) {  // plan no routed work: every weight row read stays in range
      rs.U = 0;
      atomicOr(a.err, kErrBadSlot);
    }
    if (blockIdx.x == 0) {
      PlanView P(a.plan, E);
      P.hdr[0] = V;  // routed experts only
      P.hdr[4] = 1;
    }
  }
  route_bar_sync(T);
}

// ---------------------------------------------------------------- the kernel
// Shared-memory carve-up (all offsets multiples of 16 bytes):
//   stages[NS][stage_bytes] | xq_s[T][d] | xs_s[T][d/32] | part[3][32][KS][2][2] |
//   desc[8] | full[8] | empty[8] | route_bar, go_bar | SharedCtl | RouteSmem
// The routing scores (selection scores and p(l), [T][E] each) live in the part[]
// region, which is sized for both: they are read only before the consumer
// barrier that ends the routing, and part[] is written only after it.
// NT: token count known at compile time (1 or 2): the one-token kernel has no
// second-row code.  TAPS: also store the block dots of the tapped features
// (MOE_FLAG_DEBUG_TAPS), from the same dp4a results the outputs are built from.
template <int NT, bool TAPS>
__global__ void __launch_bounds__(kThreads, 1) k_decode_fused(const FusedArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t T = NT, d = a.d, nb = d / 32, fmax = a.fmax;
  const uint32_t NS = a.n_stages;
  uint8_t *stages = smem;
  int8_t *xq_s = (int8_t *)(stages + (size_t)NS * a.stage_bytes);
  float *xs_s = (float *)(xq_s + (size_t)NT * d);
  float *part = xs_s + (size_t)NT * nb;  // [2][feature 32][K part][row 2][g,u]
  StageDesc *desc = (StageDesc *)((uint8_t *)part + a.part_bytes);
  uint64_t *full = (uint64_t *)(desc + kMaxStages);
  uint64_t *empty = full + kMaxStages;
  uint64_t *route_bar = empty + kMaxStages;  // the consumers' routing is in RouteSmem
  uint64_t *go_bar = route_bar + 1;          // the CTA's routing inputs are loaded
  SharedCtl &ctl = *(SharedCtl *)(route_bar + 2);
  volatile int *s_abort = &ctl.abort;
  int *item_cnt = ctl.item_cnt;
  RouteSmem &rs = *(RouteSmem *)(&ctl + 1);
  float *route_scratch = part;                           // [T][E] selection scores
  float *route_sig = route_scratch + (size_t)NT * a.E;  // [T][E] scores p(l)

  const SyncView SV(a.sync, a.E);
  unsigned long long *tr = a.trace ? a.trace + (size_t)blockIdx.x * kTraceWords : nullptr;
  // The consumers' inputs are loaded first, before the set-up barrier: the
  // routing inputs (a consumer thread's first logit and bias) and every x quad
  // a quantising warp will take (lane l: floats 4l..4l+3 of quad q), so that
  // each is one round trip from the kernel's start.
  const uint32_t n_quad = NT * nb / 4;  // d % 256 == 0: whole quads per token
  const uint32_t xw = (uint32_t)kConsumerWarps - NT;  // quantising warps
  const uint32_t rw = (uint32_t)(warp - kRouteWarp0);  // routing warp index (token)
  const uint32_t xi = (uint32_t)warp < (uint32_t)kRouteWarp0 ? warp : warp - NT;  // 0..xw-1
  float pre_l = 0.0f, pre_b = 0.0f;
  constexpr int kXQuads = x_quads<NT>();
  float4 xa[kXQuads];
  if (warp < kConsumerWarps) {
    if ((uint32_t)tid < NT * a.E) {
      if (!a.wr) pre_l = __ldg(a.logits + tid);
      pre_b = __ldg(a.bias + (uint32_t)tid % a.E);
    }
    const float4 *x4 = reinterpret_cast<const float4 *>(a.x);
#pragma unroll
    for (int i = 0; i < kXQuads; ++i) {
      const uint32_t q = xi + (uint32_t)i * xw;
      xa[i] = rw >= NT && q < n_quad ? __ldg(x4 + (size_t)q * 32 + lane)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (tr && tid == 0) {
    for (int i = 0; i < kTraceWords; ++i) tr[i] = 0;
    tr[kTrStart] = global_ns();
  }
  if (tid == 0) {
    // the error word is never cleared here: kernels only set bits in it and
    // moe_check_device_error clears it (a clear by one CTA could erase a bit
    // another CTA of the same call had already set)
    for (uint32_t i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    mbar_init(route_bar, 1);
    mbar_init(go_bar, 1);
    ctl.abort = ctl.writers_done = 0;
    ctl.gen = __ldcg(SV.gen);  // every CTA reads it before any can pass the exit barrier
    for (int i = 0; i < kPartBufs; ++i) ctl.item_cnt[i] = 0;
    ctl.pub_head = ctl.pub_tail = 0;
    for (int i = 0; i < kPubCap; ++i) ctl.pub_seq[i] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const uint32_t n_sh = a.fs_on / kBItemFeat;  // shared-expert gate/up items
  const uint32_t fb = a.f / kBItemFeat;      // gate/up items per routed expert

  if (warp == kProducerWarp) {
    // ============================ producer (lane 0; the warp's other lanes wait at the end)
    if (lane == 0) {
      uint32_t g = 0;  // stages issued
      bool routed = false;
      uint32_t U = 0, NB = 0, total = 0;
      unsigned long long p_wait_empty = 0, p_wait_route = 0, p_items = 0, p_wait_ready = 0;
      long long lat_ig = 0, lat_gr = 0, lat_re = 0, lat_n = 0;
      // queue order: shared gate/up | routed gate/up | shared down | routed down.
      // Only the shared gate/up items are known before routing.
      const uint32_t n_pre = n_sh;
      // wait for this CTA's consumers to finish routing (RouteSmem)
      auto learn_routing = [&]() -> bool {
        const long long t_rw = clock64();
        const bool ok = mbar_wait(route_bar, 0u, a.wait_cycles);
        p_wait_route += clock64() - t_rw;
        if (!ok) {
          report_timeout(a, 1, 0);
          *s_abort = 1;
          return false;
        }
        if (tr) tr[kTrRouteDone] = global_ns();
        U = (uint32_t)rs.U;
        NB = n_sh + U * fb;  // all gate/up items
        total = NB + (U + (a.fs_on ? 1u : 0u)) * a.n_chunks;
        routed = true;
        return true;
      };
      uint32_t item = atomicAdd(SV.queue, 1u);
      // with the router in the kernel, the weight stream starts once this CTA's
      // router loads have landed, so that they do not queue behind the stream's
      // copies in the memory system (the grid waits for the slowest CTA's)
      if (a.wr && !mbar_wait(go_bar, 0u, a.wait_cycles)) {
        report_timeout(a, 1, 1);
        *s_abort = 1;
      }
      for (;;) {
        // ticket for the following item, fetched while this one is issued
        const uint32_t next_item = atomicAdd(SV.queue, 1u);
        ++p_items;
        if (!routed && item >= n_pre && !learn_routing()) {
          *s_abort = 1;
        }
        const bool end = *s_abort || (routed && item >= total);
        StageDesc dsc;
        dsc.kind = kKindEnd;
        int nsub = 1;
        if (!end) {
          // shared-expert gate/up items come first and are known before routing
          // (NB is only known after it), so test them against n_sh before NB
          bool is_b = false, shared = false;
          uint32_t u = 0, chunk = 0;
          if (item < n_sh) {
            is_b = shared = true;
            dsc.item_first = (int)(item * kBItemFeat);
          } else if (item < NB) {
            is_b = true;
            u = (item - n_sh) / fb;
            dsc.item_first = (int)(((item - n_sh) % fb) * kBItemFeat);
          } else {
            uint32_t uc = (item - NB) / a.n_chunks;
            chunk = (item - NB) % a.n_chunks;
            if (a.fs_on && uc == 0) shared = true;
            else u = a.fs_on ? uc - 1 : uc;
          }
          if (shared) {
            dsc.e = (int)a.E;
            dsc.nrows = (int)T;
            for (uint32_t r = 0; r < T; ++r) {
              dsc.slot[r] = (int)(a.R + r);
              dsc.tok[r] = (int)r;
            }
          } else {
            dsc.e = rs.act_e[u];
            dsc.we = rs.act_w[u];
            const int row0 = rs.act_row0[u];
            dsc.nrows = rs.act_rows[u];
            for (int r = 0; r < dsc.nrows; ++r) {
              dsc.slot[r] = row0 + r;
              dsc.tok[r] = rs.tok[row0 + r];
            }
          }
          if (is_b) {
            dsc.kind = kKindB;
            nsub = kBItemFeat / kBFeat;
          } else {
            dsc.kind = kKindC;
            dsc.item_first = (int)chunk;
            dsc.first = (int)(chunk * a.c_rows);
            dsc.count = (int)min(a.c_rows, d - chunk * a.c_rows);
          }
        }
        for (int sub = 0; sub < nsub; ++sub) {
          const uint32_t st = g % NS, use = g / NS;
          const long long t_we = clock64();
          const bool empty_ok =
              use == 0 || mbar_wait(&empty[st], (use - 1) & 1u, a.wait_cycles);
          p_wait_empty += clock64() - t_we;
          if (tr && use > 0 && empty_ok) {
            lat_ig += ctl.t_got[st] - ctl.t_issue[st];
            lat_gr += ctl.t_rel[st] - ctl.t_got[st];
            lat_re += clock64() - ctl.t_rel[st];
            ++lat_n;
          }
          if (!empty_ok) {
            report_timeout(a, 2, g);
            *s_abort = 1;
            dsc.kind = kKindEnd;
          }
          dsc.sub = sub;
          uint8_t *buf = stages + (size_t)st * a.stage_bytes;
          if (dsc.kind == kKindB) {
            dsc.first = dsc.item_first + sub * kBFeat;
            dsc.count = kBFeat;
            const bool sh = dsc.e == (int)a.E;
            const size_t row = sh ? (size_t)dsc.first : (size_t)dsc.we * a.f + dsc.first;
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
            if (tr) ctl.t_issue[st] = clock64();
          } else if (dsc.kind == kKindC) {
            const bool sh = dsc.e == (int)a.E;
            const uint32_t K = sh ? a.fs : a.f;
            const size_t row = sh ? (size_t)dsc.first : (size_t)dsc.we * d + dsc.first;
            const int8_t *q_src = (sh ? a.sdq : a.dq) + row * K;
            const uint16_t *s_src = (sh ? a.sds : a.ds) + row * (K / 32);
            const uint32_t qb = (uint32_t)dsc.count * K, sb = (uint32_t)dsc.count * (K / 32) * 2;
            // the expert's h codes travel with its down weights.  The weights go
            // first (expected bytes raised without arriving, so the phase cannot
            // complete early); the h codes follow once every gate/up item of the
            // expert is published, together with the stage's single arrival.
            desc[st] = dsc;
            mbar_add_tx(&full[st], qb + sb);
            bulk_g2s(buf, q_src, qb, &full[st]);
            bulk_g2s(buf + qb, s_src, sb, &full[st]);
            if (tr) ctl.t_issue[st] = clock64();
            const long long t_wr = clock64();
            const uint32_t need = (K / kBItemFeat);
            bool ready_ok = false;
            for (int it = 0; it < kSpinIters; ++it) {
              if (ld_acquire(&SV.ready[dsc.e]) >= need) {
                ready_ok = true;
                break;
              }
              if (clock64() - t_wr > a.wait_cycles) break;
              __nanosleep(64);
            }
            p_wait_ready += clock64() - t_wr;
            if (!ready_ok) {
              // the consumers get an END stage once the weights have landed
              report_timeout(a, 4, ((uint32_t)dsc.e << 16) | __ldcg(&SV.ready[dsc.e]));
              *s_abort = 1;
              dsc.kind = kKindEnd;
              desc[st] = dsc;
              mbar_arrive(&full[st]);
              ++g;
              break;
            }
            // async-proxy reads of data that other CTAs wrote with generic stores
            asm volatile("fence.proxy.async.global;" ::: "memory");
            const uint32_t hb = K, hsb = (K / 32) * 4;
            uint8_t *hq_dst = buf + qb + sb;
            uint8_t *hs_dst = hq_dst + (size_t)kMaxT * hb;
            mbar_expect_tx(&full[st], (uint32_t)dsc.nrows * (hb + hsb));
            for (int r = 0; r < dsc.nrows; ++r) {
              const size_t slot = (size_t)(r == 0 ? dsc.slot[0] : dsc.slot[kMaxT - 1]);
              bulk_g2s(hq_dst + (size_t)r * hb, a.hq + slot * fmax, hb, &full[st]);
              bulk_g2s(hs_dst + (size_t)r * hsb, a.hs + slot * (fmax / 32), hsb, &full[st]);
            }
          } else {
            desc[st] = dsc;
            mbar_arrive(&full[st]);
          }
          ++g;
          if (dsc.kind == kKindEnd) break;
        }
        if (dsc.kind == kKindEnd) break;
        item = next_item;
      }
      atomicAdd(&ctl.writers_done, 1);  // the producer posts no events
      if (tr) {
        tr[kTrProdEnd] = global_ns();
        tr[kTrWaitEmpty] = p_wait_empty;
        tr[kTrWaitRoute] = p_wait_route;
        tr[kTrItems] = p_items;
        tr[kTrWaitReady] = p_wait_ready;
        tr[kTrLatIssueGot] = lat_ig;
        tr[kTrLatGotRel] = lat_gr;
        tr[kTrLatRelEmpty] = lat_re;
        tr[kTrLatSamples] = lat_n;
      }
    }
    __syncwarp();
  } else if (warp == kPublisherWarp) {
    // ============================ publisher (lane 0): takes the CTA's events in
    // order and does their gpu-scope release adds to the experts' readiness
    // counts (the requantising warp's stores were ordered before the event by a
    // CTA-scope fence), so that no producer or consumer warp waits on them
    if (lane == 0) {
      const long long t_pub = clock64();
      unsigned long long busy = 0;
      for (int i = 0;; ++i) {
        bool have = false;
        const long long t0 = clock64();
        for (int it = 0; it < kSpinIters; ++it) {
          if (*(volatile int *)&ctl.pub_seq[i % kPubCap] == i + 1) {
            have = true;
            break;
          }
          if (*(volatile int *)&ctl.writers_done == kConsumerWarps + 1 &&
              i >= *(volatile int *)&ctl.pub_head)
            break;
          if (clock64() - t0 > a.wait_cycles) {
            report_timeout(a, 6, (uint32_t)i);
            *s_abort = 1;
            break;
          }
          __nanosleep(256);
        }
        if (!have) break;
        __threadfence_block();
        const long long t1 = clock64();
        const int ev = ctl.pub_ev[i % kPubCap];
        *(volatile int *)&ctl.pub_tail = i + 1;
        red_release_add(&SV.ready[ev], 1u);
        busy += clock64() - t1;
      }
      if (tr) tr[kTrRouteTopk] = busy;
      (void)t_pub;
    }
    __syncwarp();
  } else {
    // ============================ consumers (warps 0..15)
    // x: every CTA quantises it for itself (CTA 0 also publishes xq/xs).  A warp
    // load covers a quad of 4 blocks (lane l: floats 4l..4l+3, block l/8); the
    // warps that do not route take quads round-robin (loaded at entry) in a
    // compact rolled loop (the code runs once per call, with a cold cache).
    auto quant_quad = [&](uint32_t q, float4 v) {
      float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll 1
      for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float sc = __fdiv_rn(amax, 127.0f);
      const uint32_t packed = (uint32_t)(uint8_t)quant_one(v.x, sc) |
                              ((uint32_t)(uint8_t)quant_one(v.y, sc) << 8) |
                              ((uint32_t)(uint8_t)quant_one(v.z, sc) << 16) |
                              ((uint32_t)(uint8_t)quant_one(v.w, sc) << 24);
      const size_t e0 = (size_t)q * 128 + 4 * lane;  // first element of this lane
      *reinterpret_cast<uint32_t *>(xq_s + e0) = packed;
      if ((lane & 7) == 0) xs_s[q * 4 + lane / 8] = sc;
      if (blockIdx.x == 0) {
        *reinterpret_cast<uint32_t *>(a.xq + e0) = packed;
        if ((lane & 7) == 0) a.xs[q * 4 + lane / 8] = sc;
      }
    };
    if (a.wr) {
      // router logits: the (expert, segment) units are spread over every
      // consumer warp of the grid, each writing its segment's partial sums for
      // the T tokens; then the CTA counts itself in and waits for all CTAs
      // (all are resident and each arrives before it waits, so the wait ends)
      const uint32_t units = a.E * a.nseg, n_warps = gridDim.x * kConsumerWarps;
      const float *xr[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) xr[t] = a.x + (size_t)t * d;
#pragma unroll 1
      for (uint32_t u = (uint32_t)warp * gridDim.x + blockIdx.x; u < units; u += n_warps) {
        const uint32_t e = u / a.nseg, g = u % a.nseg;
        float p[NT];
        router_seg_sums<NT, NT == 1 ? 32 : 16>(xr, a.wr + (size_t)e * d, g, d, lane, p);
        if (lane == 0) {
#pragma unroll
          for (int t = 0; t < NT; ++t) a.rseg[((size_t)t * a.E + e) * a.nseg + g] = p[t];
        }
      }
      consumer_sync();
      if (tid == 0) {
        mbar_arrive(go_bar);
        red_release_add(SV.queue + 1, 1u);
        if (tr) tr[27] = global_ns();
        const long long t0 = clock64();
        for (int i = 0;; ++i) {
          const uint32_t n = ld_acquire(SV.queue + 1);
          if (n >= gridDim.x) break;
          if (i >= kSpinIters || clock64() - t0 > a.wait_cycles) {
            report_timeout(a, 7, n);
            *s_abort = 1;
            break;
          }
        }
      }
      consumer_sync();
    }
    // every consumer thread scores a share of the T*E pairs (one compact
    // rolled loop: this code runs once per call with a cold instruction cache,
    // where a warp scoring a whole token in unrolled code was slower)
    route_scores(a, route_scratch, route_sig, pre_l, pre_b);
    consumer_sync();
    if (tr && tid == 0) tr[kTrRouteLoaded] = global_ns();
    if (rw < T) {
      route_select(a, rs, route_scratch, route_sig, tr);
      if (tr && rw == 0 && lane == 0) tr[kTrRoutePerm] = global_ns();
      if (rw == 0 && lane == 0 && !a.stall_test) mbar_arrive(route_bar);  // routed items may go
    } else {
      // rolled; the quads shift down one register each pass (static indices
      // keep them in registers)
#pragma unroll 1
      for (uint32_t q = xi; q < n_quad; q += xw) {
        quant_quad(q, xa[0]);
#pragma unroll
        for (int i = 0; i + 1 < kXQuads; ++i) xa[i] = xa[i + 1];
      }
    }
    consumer_sync();
    if (tr && tid == 0) tr[kTrXqDone] = global_ns();

    // trace accumulators live in registers; written once when the consumers leave
    unsigned long long c_wait_full = 0, c_b = 0, c_c = 0, n_b = 0, n_c = 0, c_item = 0;
    // gate/up: warp w takes feature w / kKSplit of the stage, K part w % kKSplit
    const uint32_t half = warp % kKSplit, fw = warp / kKSplit;
    const uint32_t nbh = nb / kKSplit;  // 32-blocks per K part
    const uint32_t nc = d / (16 * kKSplit);  // 16-byte chunks per K part
    // one token: the warp's K part of x never changes, so its codes and block
    // scales stay in registers for every gate/up stage (lane: chunks lane + 32i)
    uint4 xr[kXRegs];
    float xsr[kXRegs];
    if (NT == 1) {
#pragma unroll
      for (int i = 0; i < kXRegs; ++i) {
        const uint32_t c = lane + 32u * i;
        const bool ok = c < nc;
        xr[i] = ok ? lds16(xq_s + (size_t)half * (d / kKSplit) + 16 * c) : make_uint4(0, 0, 0, 0);
        xsr[i] = ok ? xs_s[half * nbh + (c >> 1)] : 0.0f;
      }
    }
    uint32_t b_items = 0;  // gate/up items finished by this CTA (part[] buffer parity)
    uint32_t g = 0;
    for (;; ++g) {
      const uint32_t st = g % NS, use = g / NS;
      const long long t_wf = clock64();
      const bool full_ok = mbar_wait(&full[st], use & 1u, a.wait_cycles);
      const long long t_got = clock64();
      if (tr && tid == 0) ctl.t_got[st] = t_got;
      c_wait_full += t_got - t_wf;
      if (tr && tid == 0 && g == 0) tr[kTrFirstStage] = global_ns();
      if (!full_ok) {
        report_timeout(a, 3, g);
        break;
      }
      const StageDesc dsc = desc[st];
      if (dsc.kind == kKindEnd) break;
      const uint8_t *buf = stages + (size_t)st * a.stage_bytes;
      const int nr = NT == 1 ? 1 : dsc.nrows;
      const int tok0 = dsc.tok[0], tok1 = dsc.tok[kMaxT - 1];
      if (dsc.kind == kKindB) {
        // ---- gate/up: kKSplit warps split feature first+f over K.  Lane l reads
        // 16 contiguous bytes (conflict-free): half of a 32-block, whose exact
        // int32 sum the lane scales itself (the pair's halves meet in the warp
        // sum: the same terms as a whole-block sum, another fp32 order).
        const size_t hoff = (size_t)half * (d / kKSplit);  // byte offset of this warp's K part
        const int8_t *gc = (const int8_t *)buf + (size_t)fw * d + hoff;
        const int8_t *uc = (const int8_t *)buf + (size_t)kBFeat * d + (size_t)fw * d + hoff;
        const uint16_t *gsc =
            (const uint16_t *)(buf + 2 * kBFeat * d) + (size_t)fw * nb + half * nbh;
        const uint16_t *usc = (const uint16_t *)(buf + 2 * kBFeat * d) + (size_t)kBFeat * nb +
                              (size_t)fw * nb + half * nbh;
        const int8_t *x0p = xq_s + (size_t)tok0 * d + hoff;
        const int8_t *x1p = xq_s + (size_t)tok1 * d + hoff;
        const float *xs0p = xs_s + tok0 * nb + half * nbh;
        const float *xs1p = xs_s + tok1 * nb + half * nbh;
        float g0 = 0.0f, u0 = 0.0f, g1 = 0.0f, u1 = 0.0f;
        // taps: this warp's feature, if tapped; rows' tap entries of block b at
        // tg0 / tg1 + b (gate), + kNTap * nb (up)
        int jt = -1;
        int32_t *tg0 = nullptr, *tg1 = nullptr;
        if (TAPS) {
          jt = tapped((uint32_t)(dsc.first + (int)fw), dsc.e == (int)a.E ? a.fs : a.f);
          if (jt >= 0) {
            tg0 = a.tap_gu + ((size_t)dsc.slot[0] * 2 * kNTap + jt) * nb + half * nbh;
            tg1 = a.tap_gu + ((size_t)dsc.slot[kMaxT - 1] * 2 * kNTap + jt) * nb + half * nbh;
          }
        }
        if (NT == 1) {
          // x from registers: only the weights and their scales come from the stage
#pragma unroll
          for (int i = 0; i < kXRegs; ++i) {
            if (32u * i < nc) {  // warp-uniform
              const uint32_t c = lane + 32u * i;
              const bool ok = c < nc;
              const uint4 z = make_uint4(0, 0, 0, 0);
              const uint4 wg = ok ? lds16(gc + 16 * c) : z, wu = ok ? lds16(uc + 16 * c) : z;
              const int pg = dot16(wg, xr[i]), pu = dot16(wu, xr[i]);
              const uint32_t blk = ok ? c >> 1 : 0;
              if (TAPS && jt >= 0) {
                const int bg = pair_sum(pg, lane), bu = pair_sum(pu, lane);
                if (ok && !(lane & 1)) {
                  tg0[blk] = bg;
                  tg0[blk + (size_t)kNTap * nb] = bu;
                }
              }
              const float sg = half_bits_to_float(gsc[blk]), su = half_bits_to_float(usc[blk]);
              if (ok) {
                g0 = __fmaf_rn((float)pg, sg * xsr[i], g0);
                u0 = __fmaf_rn((float)pu, su * xsr[i], u0);
              }
            }
          }
        } else {
#pragma unroll 2
        for (uint32_t c = lane; c < nc; c += 32) {
          const uint4 wg = lds16(gc + 16 * c), wu = lds16(uc + 16 * c);
          const uint32_t blk = c >> 1;
          const float sg = half_bits_to_float(gsc[blk]), su = half_bits_to_float(usc[blk]);
          const uint4 x0 = lds16(x0p + 16 * c);
          const float xs0 = xs0p[blk];
          const int pg0 = dot16(wg, x0), pu0 = dot16(wu, x0);
          g0 = __fmaf_rn((float)pg0, sg * xs0, g0);
          u0 = __fmaf_rn((float)pu0, su * xs0, u0);
          if (TAPS && jt >= 0) {
            const int bg = pair_sum(pg0, lane), bu = pair_sum(pu0, lane);
            if (!(lane & 1)) {
              tg0[blk] = bg;
              tg0[blk + (size_t)kNTap * nb] = bu;
            }
          }
          if (nr > 1) {
            const uint4 x1 = lds16(x1p + 16 * c);
            const float xs1 = xs1p[blk];
            const int pg1 = dot16(wg, x1), pu1 = dot16(wu, x1);
            g1 = __fmaf_rn((float)pg1, sg * xs1, g1);
            u1 = __fmaf_rn((float)pu1, su * xs1, u1);
            if (TAPS && jt >= 0) {
              const int bg = pair_sum(pg1, lane), bu = pair_sum(pu1, lane);
              if (!(lane & 1)) {
                tg1[blk] = bg;
                tg1[blk + (size_t)kNTap * nb] = bu;
              }
            }
          }
        }
        }
        // warp sums of (g0, u0) [, (g1, u1)] in one butterfly: the first step(s)
        // hand each lane half (quarter) one of the values, then 4 (3) steps
        // finish them; the sums land in lanes 0, 16 [, 8, 24]
        float red;
        if (NT > 1 && nr > 1) {
          const bool lo = lane < 16;
          float x0 = (lo ? g0 : u0) + __shfl_xor_sync(0xffffffffu, lo ? u0 : g0, 16);
          float x1 = (lo ? g1 : u1) + __shfl_xor_sync(0xffffffffu, lo ? u1 : g1, 16);
          const bool lo8 = (lane & 8) == 0;
          red = (lo8 ? x0 : x1) + __shfl_xor_sync(0xffffffffu, lo8 ? x1 : x0, 8);
#pragma unroll
          for (int o = 4; o > 0; o >>= 1) red += __shfl_xor_sync(0xffffffffu, red, o);
        } else {
          const bool lo = lane < 16;
          red = (lo ? g0 : u0) + __shfl_xor_sync(0xffffffffu, lo ? u0 : g0, 16);
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) red += __shfl_xor_sync(0xffffffffu, red, o);
        }
        // partial sums [feature][K part][row][g, u] in buffer b_items % kPartBufs
        // (see kPartBufs: the requant of an item never races the refill)
        const uint32_t pb = b_items % kPartBufs;
        float *pbuf = part + (size_t)pb * kBItemFeat * kKSplit * kMaxT * 2;
        {
          float *pp =
              pbuf + ((size_t)((dsc.first - dsc.item_first) + fw) * kKSplit + half) * kMaxT * 2;
          if (NT > 1 && nr > 1) {
            // lane 0: g0, 8: g1, 16: u0, 24: u1
            if ((lane & 7) == 0) pp[((lane >> 3) & 1) * 2 + (lane >> 4)] = red;
          } else {
            if ((lane & 15) == 0) pp[lane >> 4] = red;
          }
        }
        // the stage's data is no longer needed: release it before the item's
        // requant, so that the producer can refill the slot meanwhile
        __syncwarp();
        if (tr && tid == 0) ctl.t_rel[st] = clock64();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (dsc.sub == kBItemFeat / kBFeat - 1) {
          const long long t_item = clock64();
          // the item's 32 features: the last warp to finish its part computes
          // h = silu(g)*u and requantises it (lane = feature), then raises the
          // expert's readiness count (gpu-scope release) -- no warp waits
          int last = 0;
          if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&item_cnt[pb], 1) == kConsumerWarps - 1;
            if (last) {
              item_cnt[pb] = 0;
              __threadfence_block();
            }
          }
          if (__shfl_sync(0xffffffffu, last, 0)) {
            __syncwarp();
            const float *pp = pbuf + (size_t)lane * kKSplit * kMaxT * 2;
            for (int r = 0; r < nr; ++r) {
              float gv = pp[r * 2], uv = pp[r * 2 + 1];
#pragma unroll
              for (int q = 1; q < kKSplit; ++q) {
                gv = __fadd_rn(gv, pp[q * kMaxT * 2 + r * 2]);
                uv = __fadd_rn(uv, pp[q * kMaxT * 2 + r * 2 + 1]);
              }
              const float v = __fmul_rn(__fdiv_rn(gv, __fadd_rn(1.0f, spec_exp(-gv))), uv);
              float amax = fabsf(v);
#pragma unroll
              for (int o = 16; o > 0; o >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
              const float sc = __fdiv_rn(amax, 127.0f);
              const size_t slot = (size_t)(r == 0 ? dsc.slot[0] : dsc.slot[kMaxT - 1]);
              a.hq[slot * fmax + dsc.item_first + lane] = (int8_t)quant_one(v, sc);
              if (lane == 0) a.hs[slot * (fmax / 32) + dsc.item_first / 32] = sc;
            }
            __syncwarp();
            if (lane == 0) pub_post(a, ctl, dsc.e);  // the publisher raises ready[e]
          }
          ++b_items;
          c_item += clock64() - t_item;
        }
        n_b += 1;
        c_b += clock64() - t_got;
      } else {
        // ---- down: the stage holds the rows' weights and the expert's h codes
        const bool sh = dsc.e == (int)a.E;
        const uint32_t K = sh ? a.fs : a.f, kb = K / 32;
        const int8_t *hq_st = (const int8_t *)buf + (size_t)dsc.count * (K + K / 16);
        const float *hs_st = (const float *)(hq_st + (size_t)kMaxT * K);
        const int8_t *qc = (const int8_t *)buf;
        const uint16_t *scl = (const uint16_t *)(buf + (size_t)dsc.count * K);
        const size_t slot0 = (size_t)dsc.slot[0], slot1 = (size_t)dsc.slot[kMaxT - 1];
        const uint32_t ncr = K / 16;  // 16-byte chunks per down row
        // rows m0, m0+16, .. of the stage: each h chunk is read once for kDnRows rows
        for (int m0 = warp; m0 < dsc.count; m0 += kDnRows * kConsumerWarps) {
          float acc[kDnRows][kMaxT];
#pragma unroll
          for (int j = 0; j < kDnRows; ++j) acc[j][0] = acc[j][1] = 0.0f;
          // taps: the tap index of each of the warp's rows (-1: not tapped)
          int jtd[kDnRows];
#pragma unroll
          for (int j = 0; j < kDnRows; ++j) {
            const int m = m0 + j * kConsumerWarps;
            jtd[j] = TAPS && m < dsc.count ? tapped((uint32_t)(dsc.first + m), d) : -1;
          }
          for (uint32_t c0 = 0; c0 < ncr; c0 += 32) {
            const uint32_t c = c0 + lane;
            const bool ok = c < ncr;
            const uint32_t blk = ok ? c >> 1 : 0;
            const uint4 z = make_uint4(0, 0, 0, 0);
            const uint4 h0 = ok ? lds16(hq_st + 16 * c) : z;
            const float hs0 = hs_st[blk];
            uint4 h1 = z;
            float hs1 = 0.0f;
            if (nr > 1) {
              h1 = ok ? lds16(hq_st + K + 16 * c) : z;
              hs1 = hs_st[kb + blk];
            }
#pragma unroll
            for (int j = 0; j < kDnRows; ++j) {
              const int m = m0 + j * kConsumerWarps;
              const bool live = ok && m < dsc.count;
              const uint4 wd = live ? lds16(qc + (size_t)m * K + 16 * c) : make_uint4(0, 0, 0, 0);
              const float sw = live ? half_bits_to_float(scl[(size_t)m * kb + blk]) : 0.0f;
              // each lane scales its exact half-block sum (the halves meet in
              // the warp sum below)
              const int p0 = dot16(wd, h0);
              acc[j][0] = __fmaf_rn((float)p0, sw * hs0, acc[j][0]);
              if (TAPS && jtd[j] >= 0) {
                const int b0 = pair_sum(p0, lane);
                if (ok && !(lane & 1))
                  a.tap_dn[(slot0 * kNTap + jtd[j]) * (fmax / 32) + blk] = b0;
              }
              if (nr > 1) {
                const int p1 = dot16(wd, h1);
                acc[j][1] = __fmaf_rn((float)p1, sw * hs1, acc[j][1]);
                if (TAPS && jtd[j] >= 0) {
                  const int b1 = pair_sum(p1, lane);
                  if (ok && !(lane & 1))
                    a.tap_dn[(slot1 * kNTap + jtd[j]) * (fmax / 32) + blk] = b1;
                }
              }
            }
          }
#pragma unroll
          for (int j = 0; j < kDnRows; ++j) {
            const int m = m0 + j * kConsumerWarps;
            const float v0 = warp_sum(acc[j][0]);
            const float v1 = nr > 1 ? warp_sum(acc[j][1]) : 0.0f;
            if (lane == 0 && m < dsc.count) {
              a.o[slot0 * d + dsc.first + m] = v0;
              if (nr > 1) a.o[slot1 * d + dsc.first + m] = v1;
            }
          }
        }
        __syncwarp();
        if (tr && tid == 0) ctl.t_rel[st] = clock64();
        if (lane == 0) mbar_arrive(&empty[st]);
        n_c += 1;
        c_c += clock64() - t_got;
      }
    }
    if (lane == 0) atomicAdd(&ctl.writers_done, 1);  // this warp posts no more events
    if (tr && tid == 0) {
      tr[kTrConsEnd] = global_ns();
      tr[kTrWaitFull] = c_wait_full;
      tr[kTrItemEnd] = c_item;
      tr[kTrComputeB] = c_b;
      tr[kTrComputeC] = c_c;
      tr[kTrStagesB] = n_b;
      tr[kTrStagesC] = n_c;
    }
    if (tr && warp == 5 && lane == 0) {
      tr[kTrW5WaitFull] = c_wait_full;
      tr[kTrW5ComputeB] = c_b;
      tr[kTrW5ComputeC] = c_c;
    }
  }

  // ============================ exit: combine, after every CTA's o rows are written
  // A grid barrier (all CTAs are resident and each arrives before it waits, so
  // the wait ends), then the T*d outputs are split over all threads of the
  // grid: y = o_shared + sum_j w_j o_j, shared first, then slots in order, the
  // k loads of an output issued together (one round trip).
  __syncthreads();
  if (tid == 0) {
    red_release_add(SV.fin, 1u);  // this CTA's o stores, ordered by the barrier
    const uint32_t base = ctl.gen * gridDim.x;  // fin before this call (mod 2^32)
    const long long t0 = clock64();
    for (int i = 0;; ++i) {
      const uint32_t n = ld_acquire(SV.fin) - base;
      if (n >= gridDim.x) break;
      if (i >= kSpinIters || clock64() - t0 > a.wait_cycles) {
        report_timeout(a, 0, n);
        *s_abort = 1;
        break;
      }
      __nanosleep(32);
    }
  }
  __syncthreads();
  const long long t_comb = clock64();
  if (!*s_abort) {
    constexpr uint32_t kJ = 8;
#pragma unroll 1
    for (uint32_t i = blockIdx.x * kThreads + tid; i < T * d; i += gridDim.x * kThreads) {
      const uint32_t t = i / d, m = i % d;
      float acc = a.fs_on ? __ldcg(a.o + ((size_t)a.R + t) * d + m) : 0.0f;
#pragma unroll 1
      for (uint32_t j0 = 0; j0 < a.k; j0 += kJ) {
        float v[kJ];
        bool own[kJ];
#pragma unroll
        for (uint32_t jj = 0; jj < kJ; ++jj) {
          const uint32_t r = t * a.k + j0 + jj;
          own[jj] = j0 + jj < a.k && (uint32_t)rs.idx[r] >= a.e_lo && (uint32_t)rs.idx[r] < a.e_hi;
          v[jj] = own[jj] ? __ldcg(a.o + (size_t)rs.pos[r] * d + m) : 0.0f;
        }
#pragma unroll
        for (uint32_t jj = 0; jj < kJ; ++jj)
          if (own[jj]) acc = __fmaf_rn(rs.w[t * a.k + j0 + jj], v[jj], acc);
      }
      a.y[(size_t)t * d + m] = acc;
    }
  }
  if (tr && tid == 0) tr[kTrCombine] += clock64() - t_comb;
  // Every CTA has passed the barrier above, so no CTA uses the queue, router
  // and readiness counters any more: CTA 0 zeroes them for the next call and
  // counts the call (fin is not cleared: it counts up, and the next call's
  // target follows from gen), with no atomic round trip at any CTA's exit.
  if (blockIdx.x == 0) {
    for (uint32_t i = tid; i < SV.n_clear; i += kThreads)
      if (i != 2 && i != 3) a.sync[i] = 0u;
    if (tid == 0) *(volatile uint32_t *)SV.gen = ctl.gen + 1u;
  }
  if (tr && tid == 0) tr[kTrExit] = global_ns();
}

}  // namespace

// host side --------------------------------------------------------------------
namespace {
struct FusedPlan {
  uint32_t c_rows, n_chunks, n_stages, stage_bytes, part_bytes;
  size_t smem;
};

bool fused_plan(const Ctx &c, FusedPlan *fp) {
  const moe_desc &D = c.desc;
  if (c.T < 1 || c.T > (uint32_t)kMaxT) return false;
  if (D.routed_fmt != MOE_FMT_Q8_0) return false;
  if (D.flags & MOE_FLAG_FORCE_GEMV) return false;
  if (D.flags & MOE_FLAG_FORCE_TC) return false;
  if (D.top_k > 32) return false;
  if (D.d % 256 || D.f % 256 || D.f_shared % 256) return false;
  if (D.d % (32 * kKSplit * 2)) return false;  // whole, even chunk counts per K part
  if (D.d > 16u * kKSplit * 32 * kXRegs) return false;  // x of a K part fits the registers
  if (c.R > (uint32_t)kMaxR) return false;
  if ((D.d + kRouterSeg - 1) / kRouterSeg > kMaxSeg) return false;
  const uint32_t d = D.d, fmax = c.fmax;
  const size_t b_bytes = (size_t)kBFeat * 2 * (d + d / 16);
  const uint32_t row_c = fmax + fmax / 16;
  // a down stage also carries the expert's h codes and scales (up to 2 rows)
  const size_t h_bytes = (size_t)kMaxT * (fmax + (fmax / 32) * 4);
  if (b_bytes <= h_bytes) return false;
  uint32_t c_rows = (uint32_t)((b_bytes - h_bytes) / row_c);
  if (c_rows == 0) return false;
  if (c_rows > d) c_rows = d;
  const uint32_t n_chunks = (d + c_rows - 1) / c_rows;
  if (4 + D.n_expert + 1 + 2 > kSyncInts) return false;  // ready[E+1] clear of fin, gen
  const size_t stage = (b_bytes + 127) / 128 * 128;
  size_t part = (size_t)kPartBufs * kBItemFeat * kKSplit * kMaxT * 2 * 4;
  const size_t scores = 2 * (size_t)c.T * D.n_expert * 4;
  part = (part > scores ? part : scores + 15) / 16 * 16;
  const size_t rest = (size_t)c.T * d + (size_t)c.T * (d / 32) * 4 + part +
                      kMaxStages * sizeof(StageDesc) +
                      2 * kMaxStages * 8 + 16 + sizeof(SharedCtl) + sizeof(RouteSmem) + 128;
  int dev = 0, max_smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
      cudaSuccess)
    return false;
  if ((size_t)max_smem < rest + 2 * stage) return false;
  uint32_t ns = (uint32_t)(((size_t)max_smem - rest) / stage);
  if (ns > (uint32_t)kMaxStages) ns = kMaxStages;
  fp->c_rows = c_rows;
  fp->n_chunks = n_chunks;
  fp->n_stages = ns;
  fp->stage_bytes = (uint32_t)stage;
  fp->part_bytes = (uint32_t)part;
  fp->smem = rest + ns * stage;
  return true;
}
}  // namespace

size_t fused_sync_ints(const moe_desc *d) {
  (void)d;
  return kSyncInts;
}

bool fused_eligible(const Ctx &c) {
  FusedPlan fp;
  return fused_plan(c, &fp);
}

cudaError_t launch_decode_fused(const Ctx &c, const float *x, const float *logits,
                                const float *bias, float *y, const float *w_router,
                                float *logits_out) {
  FusedPlan fp;
  if (!fused_plan(c, &fp)) return cudaErrorNotSupported;
  const moe_desc &D = c.desc;
  FusedArgs a;
  a.E = D.n_expert;
  a.k = D.top_k;
  a.d = D.d;
  a.f = D.f;
  a.fs = D.f_shared;
  a.e_lo = c.e_lo;
  a.e_hi = c.e_hi;
  a.fs_on = c.shared_on ? D.f_shared : 0u;
  a.T = c.T;
  a.R = c.R;
  a.fmax = c.fmax;
  a.s = D.s;
  a.score = D.score;
  a.x = x;
  a.logits = w_router ? nullptr : logits;
  a.bias = bias;
  a.wr = w_router;
  a.logits_out = logits_out;
  a.rseg = (float *)(c.ws + c.L.rseg);
  a.nseg = (D.d + kRouterSeg - 1) / kRouterSeg;
  if (w_router && (!c.L.rseg || !logits_out)) return cudaErrorInvalidValue;
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
  a.eslot = c.wts.expert_slot;
  a.n_slots = c.wexp;
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
  a.part_bytes = fp.part_bytes;
  a.stall_test = (D.flags & MOE_FLAG_TEST_STALL) ? 1 : 0;
  a.wait_cycles = a.stall_test ? kStallTestCycles : kWaitCycles;
  a.trace = (D.flags & MOE_FLAG_TRACE) ? (unsigned long long *)(c.ws + c.L.trace) : nullptr;
  const bool taps = (D.flags & MOE_FLAG_DEBUG_TAPS) != 0;
  if (taps && (!c.L.tap_gu || !c.L.tap_dn)) return cudaErrorInvalidValue;
  a.tap_gu = taps ? (int32_t *)(c.ws + c.L.tap_gu) : nullptr;
  a.tap_dn = taps ? (int32_t *)(c.ws + c.L.tap_dn) : nullptr;
  auto kern = c.T == 1 ? (taps ? k_decode_fused<1, true> : k_decode_fused<1, false>)
                       : (taps ? k_decode_fused<2, true> : k_decode_fused<2, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace moe
