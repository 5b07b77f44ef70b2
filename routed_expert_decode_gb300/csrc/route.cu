// route.cu -- router, permutation, work plan and activation quantiser.
//
// Router: sigmoid scoring plus a selection bias, top_k per token ("sigmoid
// routing with top-8": "256 experts, 512 lines", section "Why GLM-5.2 in an
// engine built for DeepSeek"; Hy3's "192-expert top-8 sigmoid router with expert
// bias": NeutronStar main README).  One generic warp-per-token kernel for every
// n_expert / top_k / scale: no constant is baked in (the lesson of "The constant
// that always said 256").
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;

// One warp per token.  Lane l owns experts l, l+32, ... (NPER of them: the
// kernel is instantiated for E <= 256, 512 and 1024 so that its unrolled loops
// are no longer than the layer needs -- this code runs once per call from a
// cold instruction cache); each of the top_k rounds takes every lane's best
// unpicked expert and reduces them with a butterfly argmax whose order is
// (score descending, index ascending), so all lanes agree on a unique winner
// and ties go to the lower index.
template <int NPER>
__global__ void __launch_bounds__(kRouteWarps * 32)
    k_route(const float *__restrict__ logits, const float *__restrict__ bias, uint32_t T,
            uint32_t E, uint32_t k, float s, uint32_t score, int32_t *__restrict__ idx,
            float *__restrict__ w) {
  pdl_trigger();
  pdl_wait();  // the logits may come from the router kernel before it
  const int lane = threadIdx.x & 31;
  const uint32_t t = blockIdx.x * kRouteWarps + threadIdx.x / 32;
  if (t >= T) return;
  const float *l = logits + (size_t)t * E;
  const int nper = (int)((E + 31) / 32);
  float c[NPER], sg[NPER];
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const uint32_t e = (uint32_t)lane + 32u * i;
    c[i] = -INFINITY;
    sg[i] = 0.0f;
    if (i < nper && e < E) {
      const float sgm = score_rn(l[e], score);
      sg[i] = sgm;
      c[i] = __fadd_rn(sgm, bias[e]);
    }
  }
  uint32_t taken = 0;
  float my_sigma = 0.0f;  // lane j keeps the sigma of slot j
  for (uint32_t j = 0; j < k; ++j) {
    float bc = -INFINITY, bs = 0.0f;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
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
    if (lane == 0) idx[(size_t)t * k + j] = be;
  }
  // w_j = s * sigma_j / sum_j sigma_j, the sum taken in slot order
  float sum = 0.0f;
  for (uint32_t j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, my_sigma, j));
  if ((uint32_t)lane < k) w[(size_t)t * k + lane] = __fmul_rn(s, __fdiv_rn(my_sigma, sum));
}

// Block-wide exclusive scan of one int per thread, for a block of 32 full warps
// (1024 threads): each warp scans its 32 values by shuffles, warp 0 scans the
// 32 warp totals, three barriers in all.  Returns the exclusive prefix; *total
// gets the block sum.  wsum: 32 ints of shared memory, free again on return.
__device__ int block_excl_scan(int v, int *wsum, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    wsum[lane] = t;  // inclusive prefix of the warp totals
  }
  __syncthreads();
  const int before = warp > 0 ? wsum[warp - 1] : 0;
  *total = wsum[31];
  __syncthreads();
  return before + x - v;
}

// Stable permutation without position atomics (1 CTA, 32 warps).
// Rows r = t*k + j.  Warp w owns a contiguous range of tokens; (A) each warp
// counts its rows per expert, (B) a per-expert scan over warps gives each warp's
// starting rank, (C) a scan over experts gives off[], (D) each warp walks its
// rows in order, ranking equal experts inside a 32-row group with match_any.
constexpr int kPermThreads = 1024;
static_assert(kPermThreads == 1024, "block_excl_scan takes 32 full warps");
constexpr int kPermWarps = kPermThreads / 32;

__global__ void __launch_bounds__(kPermThreads)
    k_permute(const int32_t *__restrict__ idx, uint32_t T, uint32_t E, uint32_t k,
              int32_t *__restrict__ off, int32_t *__restrict__ perm, int32_t *__restrict__ pos,
              uint32_t *err) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int smem[];
  int *hist = smem;                       // [kPermWarps][E]
  int *cnt = hist + (size_t)kPermWarps * E;  // [E]
  int *scan = cnt + E;                    // [32]: block_excl_scan's warp totals
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (uint32_t i = tid; i < (uint32_t)kPermWarps * E; i += kPermThreads) hist[i] = 0;
  __syncthreads();
  const uint32_t tok_per_warp = (T + kPermWarps - 1) / kPermWarps;
  const uint32_t r_begin = min(T, warp * tok_per_warp) * k;
  const uint32_t r_end = min(T, (warp + 1) * tok_per_warp) * k;
  // (A)
  for (uint32_t r = r_begin + lane; r < r_end; r += 32) {
    const int e = idx[r];
    if (e < 0 || (uint32_t)e >= E) {
      if (err) atomicOr(err, kErrBadIndex);
      continue;
    }
    atomicAdd(&hist[(size_t)warp * E + e], 1);
  }
  __syncthreads();
  // (B) hist[w][e] := rows of e in warps < w
  for (uint32_t e = tid; e < E; e += kPermThreads) {
    int run = 0;
    for (int w2 = 0; w2 < kPermWarps; ++w2) {
      const int v = hist[(size_t)w2 * E + e];
      hist[(size_t)w2 * E + e] = run;
      run += v;
    }
    cnt[e] = run;
  }
  __syncthreads();
  // (C) exclusive scan of cnt over experts, in chunks of kPermThreads
  int carry = 0;
  for (uint32_t base = 0; base < E; base += kPermThreads) {
    const uint32_t e = base + tid;
    const int v = e < E ? cnt[e] : 0;
    int chunk_total;
    const int excl = carry + block_excl_scan(v, scan, &chunk_total);
    if (e < E) {
      off[e] = excl;
      cnt[e] = excl;  // cnt now holds off[e]
    }
    carry += chunk_total;
  }
  if (tid == 0) off[E] = carry;
  __syncthreads();
  // (D)
  const unsigned lt_mask = (1u << lane) - 1u;
  for (uint32_t g = r_begin; g < r_end; g += 32) {
    const uint32_t r = g + lane;
    const bool live = r < r_end;
    int e = live ? idx[r] : -1;
    if (e >= (int)E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (live && e >= 0) {
      const int rank = __popc(peers & lt_mask);
      int *run = &hist[(size_t)warp * E + e];
      const int p = cnt[e] + *run + rank;
      perm[p] = (int32_t)r;
      pos[r] = p;
    }
    __syncwarp();
    // the highest lane of each peer group advances that expert's running rank
    if (live && e >= 0 && (peers >> lane) == 1u) hist[(size_t)warp * E + e] += __popc(peers);
    __syncwarp();
  }
}

constexpr int kPlanThreads = 1024;
static_assert(kPlanThreads == 1024, "block_excl_scan takes 32 full warps");
constexpr int kMaxExperts = 1024;  // moe_desc.n_expert, checked on the host

// Work plan from off[] (1 CTA).  Validates off, perm, pos and idx against one
// another; on any inconsistency it flags kErrBadOffsets / kErrBadIndex and plans
// no work (so no kernel indexes with untrusted values).  Otherwise it lists the
// active experts (dp4a list: ascending, the shared expert last; tensor-core
// list: by rows, descending), split between the dp4a path and the tensor-core
// path: experts with more than tc_min_rows rows, when
// their gate/up tiles number at least tc_min_tiles (one per SM: fewer would
// leave most SMs idle while the GEMV kernels wait behind the tensor kernel),
// else none; every row with force_tc.
__global__ void __launch_bounds__(kPlanThreads)
    k_plan(const int32_t *__restrict__ off, const int32_t *__restrict__ idx,
           const int32_t *__restrict__ perm, const int32_t *__restrict__ pos, uint32_t T,
           uint32_t E, uint32_t k, uint32_t f, uint32_t fs, uint32_t d, int tc_mode,
           uint32_t tc_min_rows, uint32_t tc_min_tiles, const int32_t *__restrict__ eslot,
           uint32_t n_slots, uint32_t e_lo, uint32_t e_hi, int shared_on, int *plan,
           uint32_t *err) {
  pdl_trigger();
  pdl_wait();
  __shared__ int scan[32];  // block_excl_scan's warp totals
  __shared__ int bad;
  __shared__ int s_off[kMaxExperts + 1];  // off[], read from global memory once
  __shared__ int s_ntc;                   // entries of the tensor-core list
  const int tid = threadIdx.x;
  const uint32_t R = T * k;
  PlanView P(plan, E);
  for (uint32_t e = tid; e <= E; e += kPlanThreads) s_off[e] = off[e];
  if (tid == 0) bad = 0;
  __syncthreads();
  if (tid == 0 && (s_off[0] != 0 || s_off[E] != (int)R)) bad = 1;
  for (uint32_t e = tid; e < E; e += kPlanThreads)
    if (s_off[e + 1] < s_off[e]) bad = 1;
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      atomicOr(err, kErrBadOffsets);
      for (int i = 0; i < 8; ++i) P.hdr[i] = 0;  // hdr[4] = 0: nothing validated
      P.item_gu[0] = 0;
      P.tc_tile_gu[0] = P.tc_tile_dn[0] = 0;
    }
    return;
  }
  // cross-check the routing arrays: slot p of expert e's segment holds a row
  // r of e with pos[r] == p, and every pos[r] points back at r
  for (uint32_t p = tid; p < R; p += kPlanThreads) {
    const int r = perm[p];
    int lo = 0, hi = (int)E;  // largest e with off[e] <= p
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= (int)p) lo = mid; else hi = mid;
    }
    if (r < 0 || (uint32_t)r >= R || idx[r] != lo || pos[r] != (int)p) bad = 2;
  }
  for (uint32_t r = tid; r < R; r += kPlanThreads) {
    const int p = pos[r];
    if (p < 0 || (uint32_t)p >= R || perm[p] != (int)r) bad = 2;
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      atomicOr(err, kErrBadIndex);
      for (int i = 0; i < 8; ++i) P.hdr[i] = 0;
      P.item_gu[0] = 0;
      P.tc_tile_gu[0] = P.tc_tile_dn[0] = 0;
    }
    return;
  }
  // rows of expert e this call computes: only the experts in [e_lo, e_hi) (the
  // share of one rank in an expert-parallel split; all of them by default)
  auto own_rows = [&](uint32_t e) -> int {
    return e >= e_lo && e < e_hi ? s_off[e + 1] - s_off[e] : 0;
  };
  // with a slot table, every selected expert this call computes must have its
  // weights in a slot
  if (eslot) {
    for (uint32_t e = tid; e < E; e += kPlanThreads)
      if (own_rows(e) > 0 && (uint32_t)eslot[e] >= n_slots) bad = 3;
    __syncthreads();
    if (bad) {
      if (tid == 0) {
        atomicOr(err, kErrBadSlot);
        for (int i = 0; i < 8; ++i) P.hdr[i] = 0;
        P.item_gu[0] = 0;
        P.tc_tile_gu[0] = P.tc_tile_dn[0] = 0;
      }
      return;
    }
  }
  if (tc_mode == 1) {
    // gate/up tiles the row rule would send to the tensor cores
    __shared__ int tc_tiles;
    if (tid == 0) {
      tc_tiles = 0;
      if (shared_on && fs > 0 && fs == f && T > tc_min_rows)
        tc_tiles = (int)(fs / kTcTileM) * (int)((T + kTcTileN - 1) / kTcTileN);
    }
    __syncthreads();
    int mine = 0;
    for (uint32_t e = tid; e < E; e += kPlanThreads) {
      const int rows = own_rows(e);
      if (rows > (int)tc_min_rows)
        mine += (int)(f / kTcTileM) * ((rows + (int)kTcTileN - 1) / (int)kTcTileN);
    }
    if (mine) atomicAdd(&tc_tiles, mine);
    __syncthreads();
    if ((uint32_t)tc_tiles < tc_min_tiles) tc_mode = 0;
  }
  auto on_tc = [&](int rows) -> bool {
    if (tc_mode == 0 || rows <= 0) return false;
    return tc_mode == 2 ? true : (uint32_t)rows > tc_min_rows;
  };
  const int ntile_n = (int)kTcTileN;
  __shared__ int rows_max;  // the most rows of any expert this call computes
  if (tid == 0) rows_max = 0;
  __syncthreads();
  int ng = 0, ntc = 0, ntile_gu = 0, total;
  for (uint32_t base = 0; base < E; base += kPlanThreads) {
    const uint32_t e = base + tid;
    const int rows = e < E ? own_rows(e) : 0;
    const bool tc = on_tc(rows);
    const int gflag = rows > 0 && !tc ? 1 : 0, tflag = tc ? 1 : 0;
    const int gu = ng + block_excl_scan(gflag, scan, &total);
    const int gtotal = total;
    const int tv = ntc + block_excl_scan(tflag, scan, &total);
    const int ttotal = total;
    const int tiles = tc ? (int)(f / kTcTileM) * ((rows + ntile_n - 1) / ntile_n) : 0;
    const int tile0 = ntile_gu + block_excl_scan(tiles, scan, &total);
    const int tiles_total = total;
    if (gflag) {
      P.act_e[gu] = (int)e;
      P.act_row0[gu] = s_off[e];
      P.act_rows[gu] = rows;
      P.item_gu[gu] = gu * (int)f;
    }
    if (tflag) {
      P.tc_e[tv] = (int)e;
      P.tc_row0[tv] = s_off[e];
      P.tc_rows[tv] = rows;
      P.tc_tile_gu[tv] = tile0;
      P.tc_tile_dn[tv] = (tile0 / (int)(f / kTcTileM)) * (int)(d / kTcTileM);
    }
    ng += gtotal;
    ntc += ttotal;
    ntile_gu += tiles_total;
    const int wmax = __reduce_max_sync(0xffffffffu, rows);
    if ((tid & 31) == 0 && wmax > 0) atomicMax(&rows_max, wmax);
  }
  __syncthreads();
  if (tid == 0) {
    const int maxrows = rows_max;
    int U = ng;
    int items = U * (int)f;
    int V = ntc;
    int tiles_gu = ntile_gu;
    const int mt = (int)(f / kTcTileM);
    int tiles_dn = mt > 0 ? (ntile_gu / mt) * (int)(d / kTcTileM) : 0;
    if (shared_on && fs > 0 && T > 0) {
      // the shared expert reads every token; the tensor path needs fs == f
      if (on_tc((int)T) && fs == f) {
        const int nt = ((int)T + ntile_n - 1) / ntile_n;
        P.tc_e[V] = (int)E;
        P.tc_row0[V] = (int)R;
        P.tc_rows[V] = (int)T;
        P.tc_tile_gu[V] = tiles_gu;
        P.tc_tile_dn[V] = tiles_dn;
        tiles_gu += (int)(fs / kTcTileM) * nt;
        tiles_dn += (int)(d / kTcTileM) * nt;
        V += 1;
      } else {
        P.act_e[U] = (int)E;
        P.act_row0[U] = (int)R;
        P.act_rows[U] = (int)T;
        P.item_gu[U] = items;
        items += (int)fs;
        U += 1;
      }
    }
    P.item_gu[U] = items;
    P.tc_tile_gu[V] = tiles_gu;
    P.tc_tile_dn[V] = tiles_dn;
    P.hdr[0] = U;
    P.hdr[1] = items;
    P.hdr[2] = U * (int)d;
    P.hdr[3] = maxrows;
    P.hdr[4] = 1;  // routing arrays validated: the combine may read pos[]
    P.hdr[5] = V;
    s_ntc = V;
    P.hdr[6] = tiles_gu;
    P.hdr[7] = tiles_dn;
  }
  __syncthreads();
  // Tensor-core experts by rows, descending (lower expert index first on equal
  // rows; the shared expert, with every token, leads).  The tensor kernels deal
  // tiles out in rounds of one per CTA, so the widest and costliest tiles go out
  // first and the narrow ones even out the CTAs' totals at the end.
  const int V = s_ntc;
  if (V > 1) {
    // (rows, expert) of every entry in shared memory while it fits
    __shared__ int key_rows[kPlanThreads], key_e[kPlanThreads];
    const bool in_smem = V <= kPlanThreads;
    if (in_smem && tid < V) {
      key_rows[tid] = P.tc_rows[tid];
      key_e[tid] = P.tc_e[tid];
    }
    __syncthreads();
    const int *rows_of = in_smem ? key_rows : P.tc_rows;
    const int *e_of = in_smem ? key_e : P.tc_e;
    for (int v = tid; v < V; v += kPlanThreads) {
      const int rv = rows_of[v], ev = e_of[v];
      int rank = 0;
      for (int u = 0; u < V; ++u) {
        const int ru = rows_of[u];
        rank += (ru > rv || (ru == rv && e_of[u] < ev)) ? 1 : 0;
      }
      P.tc_tile_dn[rank] = ev;  // scratch: the expert at its new position
    }
    __syncthreads();
    for (int r = tid; r < V; r += kPlanThreads) {
      const int e = P.tc_tile_dn[r];
      P.tc_e[r] = e;
      P.tc_row0[r] = e == (int)E ? (int)R : s_off[e];
      P.tc_rows[r] = e == (int)E ? (int)T : s_off[e + 1] - s_off[e];
    }
    __syncthreads();
    // tile prefixes in the new order (the totals do not change)
    const int mt = (int)(f / kTcTileM), dt = (int)(d / kTcTileM);
    int done = 0;
    for (int base = 0; base < V; base += kPlanThreads) {
      const int r = base + tid;
      const int tiles = r < V ? mt * ((P.tc_rows[r] + ntile_n - 1) / ntile_n) : 0;
      const int tile0 = done + block_excl_scan(tiles, scan, &total);
      if (r < V) {
        P.tc_tile_gu[r] = tile0;
        P.tc_tile_dn[r] = (tile0 / mt) * dt;
      }
      done += total;
    }
  }
}

// Activation quantiser.  A warp unit is 4 consecutive 32-blocks of x (lane l
// holds values 4l .. 4l+3 of the 128, so lanes 8j .. 8j+7 hold block j); a
// fixed grid of warps walks the units, two at a time with both units' loads
// issued first.  Per block: amax over its 32 values, scale amax / 127, codes
// as quant_one.
__device__ __forceinline__ float4 quant_load(const float *x, uint64_t u, uint32_t nblocks,
                                             int lane) {
  const uint64_t b = 4 * u + (uint64_t)(lane >> 3);
  if (b >= nblocks) return make_float4(0.f, 0.f, 0.f, 0.f);
  const float *p = x + b * 32 + 4 * (lane & 7);
  if (((uintptr_t)x & 15u) == 0) return *reinterpret_cast<const float4 *>(p);
  return make_float4(p[0], p[1], p[2], p[3]);  // the caller's x, not 16-byte aligned
}

__device__ __forceinline__ void quant_store(float4 v, uint64_t u, uint32_t nblocks, int lane,
                                            int8_t *__restrict__ xq, float *__restrict__ xs,
                                            int8_t *__restrict__ xt) {
  float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const uint64_t b = 4 * u + (uint64_t)(lane >> 3);
  if (b >= nblocks) return;
  const float sc = __fdiv_rn(a, 127.0f);
  const int q0 = quant_one(v.x, sc), q1 = quant_one(v.y, sc), q2 = quant_one(v.z, sc),
            q3 = quant_one(v.w, sc);
  const int e0 = 4 * (lane & 7);
  *reinterpret_cast<char4 *>(xq + b * 32 + e0) =
      make_char4((signed char)q0, (signed char)q1, (signed char)q2, (signed char)q3);
  // 2-bit routed weights also read the codes with each 16-code group 4x4
  // transposed: code 16g + 4j + i at byte 16g + 4i + j
  if (xt) {
    int8_t *tb = xt + b * 32;
    const int q[4] = {q0, q1, q2, q3};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = e0 + i;
      tb[(e & 16) | ((e & 3) << 2) | ((e >> 2) & 3)] = (int8_t)q[i];
    }
  }
  if ((lane & 7) == 0) xs[b] = sc;
}

__global__ void __launch_bounds__(256)
    k_quant(const float *__restrict__ x, uint32_t nblocks, int8_t *__restrict__ xq,
            float *__restrict__ xs, int8_t *__restrict__ xt) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const uint64_t units = ((uint64_t)nblocks + 3) / 4;
  const uint64_t nw = (uint64_t)gridDim.x * 8;
  for (uint64_t u = (uint64_t)blockIdx.x * 8 + threadIdx.x / 32; u < units; u += 2 * nw) {
    const float4 v0 = quant_load(x, u, nblocks, lane);
    const float4 v1 = quant_load(x, u + nw, nblocks, lane);
    quant_store(v0, u, nblocks, lane, xq, xs, xt);
    quant_store(v1, u + nw, nblocks, lane, xq, xs, xt);
  }
}

}  // namespace

cudaError_t launch_route(const Ctx &c, const float *logits, const float *bias, int32_t *idx,
                         float *w) {
  if (c.T == 0) return cudaSuccess;
  const unsigned grid = (c.T + kRouteWarps - 1) / kRouteWarps;
  const uint32_t E = c.desc.n_expert;
  auto kern = E <= 256 ? k_route<8> : E <= 512 ? k_route<16> : k_route<32>;
  const cudaError_t e = launch_k(kern, grid, kRouteWarps * 32, 0, c.stream, c.chained, logits,
                                 bias, c.T, E, c.desc.top_k, c.desc.s, c.desc.score, idx, w);
  c.chained = true;
  return e;
}

// logits[t][e] = x[t] . w_router[e] in the library's fixed order (moe.h,
// moe_router_logits): one CTA per (t, e), warp g takes the 1024-input segment
// g (lane l: fma chain over i = 1024g + l + 32j, all loads issued first), the
// lanes' sums meet over xor distances 16..1, and thread 0 adds the segment totals
// in ascending order.
__global__ void __launch_bounds__(1024)
    k_router_logits(const float *__restrict__ x, const float *__restrict__ wr, uint32_t T,
                    uint32_t E, uint32_t d, float *__restrict__ logits) {
  pdl_trigger();
  pdl_wait();
  __shared__ float seg_total[32];
  const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
  const uint32_t t = blockIdx.x / E, e = blockIdx.x % E;
  const float *const xr[1] = {x + (size_t)t * d};
  float p[1];
  router_seg_sums<1, 32>(xr, wr + (size_t)e * d, (uint32_t)g, d, lane, p);
  if (lane == 0) seg_total[g] = p[0];
  __syncthreads();
  if (threadIdx.x == 0) {
    float total = seg_total[0];
    const int nseg = (int)((d + kRouterSeg - 1) / kRouterSeg);
    for (int s = 1; s < nseg; ++s) total = __fadd_rn(total, seg_total[s]);
    logits[(size_t)t * E + e] = total;
  }
}

cudaError_t launch_router_logits(const moe_desc &d, const float *w_router, const float *x,
                                 uint32_t T, float *logits, cudaStream_t stream) {
  const uint64_t items = (uint64_t)T * d.n_expert;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffffull || d.d > 32u * kRouterSeg) return cudaErrorInvalidValue;
  const unsigned warps = (d.d + kRouterSeg - 1) / kRouterSeg;
  k_router_logits<<<(unsigned)items, warps * 32, 0, stream>>>(x, w_router, T, d.n_expert, d.d,
                                                              logits);
  return cudaGetLastError();
}

cudaError_t launch_permute(const Ctx &c, const int32_t *idx, int32_t *off, int32_t *perm,
                           int32_t *pos, uint32_t *err) {
  const uint32_t E = c.desc.n_expert;
  const size_t smem = sizeof(int) * ((size_t)kPermWarps * E + E + 32);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_permute, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  const cudaError_t e = launch_k(k_permute, 1, kPermThreads, smem, c.stream, c.chained, idx, c.T,
                                 E, c.desc.top_k, off, perm, pos, err);
  c.chained = true;
  return e;
}

cudaError_t launch_plan(const Ctx &c, const int32_t *off, const int32_t *idx,
                             const int32_t *perm, const int32_t *pos, uint32_t *err) {
  int *plan = (int *)(c.ws + c.L.plan);
  // tensor path: 0 off, 1 for experts with more than tc_min_rows_for(fmt) rows,
  // 2 forced
  const moe_desc &D = c.desc;
  if (D.n_expert > (uint32_t)kMaxExperts) return cudaErrorInvalidValue;  // s_off's size
  int tc_mode = 0;
  // the same condition under which run_ffn launches the tensor kernels
  if (c.L.xperm && tc_supported(D) && tc_weights_aligned(c))
    tc_mode = (D.flags & MOE_FLAG_FORCE_TC) ? 2 : 1;
  const cudaError_t e = launch_k(k_plan, 1, kPlanThreads, 0, c.stream, c.chained, off, idx, perm,
                                 pos, c.T, D.n_expert, D.top_k, D.f, D.f_shared, D.d, tc_mode,
                                 tc_min_rows_for(D.routed_fmt), (uint32_t)c.sm_count, c.wts.expert_slot, c.wexp,
                                 c.e_lo, c.e_hi, c.shared_on ? 1 : 0, plan, err);
  c.chained = true;
  return e;
}

cudaError_t launch_quant_x(const Ctx &c, const float *x) {
  const uint32_t nblocks = c.T * (c.desc.d / 32);
  if (nblocks == 0) return cudaSuccess;
  // a fixed grid (at most 6 CTAs of 8 warps an SM) walking 4-block units, two a
  // warp at a time
  const uint32_t units = (nblocks + 3) / 4;
  const uint32_t ctas = std::min<uint32_t>((units + 15) / 16, (uint32_t)c.sm_count * 6);
  const cudaError_t e = launch_k(k_quant, ctas, 256, 0, c.stream, c.chained, x,
                                 nblocks, (int8_t *)(c.ws + c.L.xq), (float *)(c.ws + c.L.xs),
                                 c.L.xt ? (int8_t *)(c.ws + c.L.xt) : nullptr);
  c.chained = true;
  return e;
}

}  // namespace moe
