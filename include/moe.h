/*
 * moe.h -- C ABI of the GB300 routed Mixture-of-Experts layer (libmoe.so).
 *
 * The layer (as run by the ds4 / NeutronStar engines for GLM-5.2 and Hy3):
 *   1. score every expert with sigmoid(logit) + selection bias and keep the
 *      top_k ("sigmoid routing with top-8": "256 experts, 512 lines", section
 *      "Why GLM-5.2 in an engine built for DeepSeek"; "192-expert top-8 sigmoid
 *      router with expert bias": NeutronStar main README, Hy3 paragraph), with
 *      n_expert / top_k / scale as parameters, never constants ("256 experts,
 *      512 lines", section "The constant that always said 256");
 *   2. group the token->expert rows by expert (per-expert batches: NeutronStar
 *      README, sections "MTP speculative decoding" and "Long-prompt prefill");
 *   3. quantise activations to int8 per 32-block and run each selected expert's
 *      SwiGLU FFN with int8 x int8 block dot products over block-quantised
 *      weights (the dp4a expert kernels: NeutronStar README, "What this branch
 *      adds over upstream"; Q8_0: "The model");
 *   4. add the always-on shared expert ("MoE with shared expert") and combine
 *      the routed outputs with their routing weights.
 *
 * Arithmetic contract (bit-exact parts are identical to the CPU oracle):
 *   score     c_i = fp32(sigma_i + b_i), sigma_i = fp32(1 / (1 + spec_exp(-l_i)));
 *             spec_exp: clamp to [-86, 88], n = rint(x*log2e), Cody-Waite
 *             reduction with C1 = 355/512 and C2 = fp32(ln2 - C1), degree-7
 *             Taylor polynomial (fp32 coefficients 1/k!, Horner with fma), times
 *             2^n -- all fp32 round-to-nearest.
 *   top-k     largest c first, equal c -> lower expert index first.
 *   weights   w_j = s * sigma_j / sum_j sigma_j (fp32; not bit-exact).
 *   permute   off[e] = rows before expert e; rows of one expert in (token, slot)
 *             order: perm[off[e] + r] = t*top_k + j; pos is perm's inverse.
 *   quantise  per 32-block: scale = max|x| / 127 (fp32), q = clamp(
 *             round_half_away(x / scale), -127, 127); a zero scale gives q = 0.
 *   expert    g = sum_b isum_b * ws_b * xs_b (isum_b exact int32), likewise u;
 *             h = g * sigmoid(g) * u requantised as above; o likewise with the
 *             down matrix.  Only isum_b and the int8 x codes are bit-exact; h codes
 *             may differ by one step where fp32 order matters.
 *   combine   y[t] = o_shared[t] + sum_j w[t,j] * o[t,j], shared first, then
 *             slots in order (no atomics: run-to-run deterministic).
 *
 * Memory: every pointer is caller-owned DEVICE memory except the desc/weights
 * structs (host).  The layer entry points allocate nothing; the one object
 * that owns memory is an expert cache (moe_cache_create: host memory and CUDA
 * events, including the pinned buffer moe_stream_layer reads the picks back
 * into, freed by moe_cache_destroy).  Scratch comes from the caller's
 * workspace (moe_workspace_size).  Calls are asynchronous on `stream`
 * (a cudaStream_t; NULL = legacy default stream), stateless and re-entrant as
 * long as concurrent calls use different workspaces.  Arguments are checked on
 * the host before anything is enqueued; nothing aborts or exits.  Device-side
 * argument faults (an expert index out of range in moe_ffn's inputs) and
 * timed-out waits set bits in an error word in the workspace; kernels only ever
 * set bits, and moe_check_device_error reads and clears them.
 * NaN or infinite inputs are unsupported.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* bad shape, null or misaligned pointer */
  MOE_ERR_UNSUPPORTED = 2,  /* valid request this library does not implement */
  MOE_ERR_WORKSPACE = 3,    /* ws_bytes < moe_workspace_size() */
  MOE_ERR_CUDA = 4,         /* a CUDA launch or runtime call failed */
  MOE_ERR_TIMEOUT = 5,      /* a bounded device wait gave up */
  MOE_ERR_DEVICE_CHECK = 6  /* the kernels flagged a bad input on the device */
} moe_status;

/* Weight formats, both planar: a code plane and an fp16 scale plane, one scale
 * per 32 consecutive weights along the reduction dimension.
 *   MOE_FMT_Q8_0: int8 codes, row of K weights = K bytes + K/32 fp16.
 *   MOE_FMT_Q2S : 2-bit codes c in {0,1,2,3} meaning {-3,-1,+1,+3}; weight i of
 *                 a row sits at bits 2(i%4) of byte i/4 (LSB first); a row of K
 *                 weights = K/4 bytes + K/32 fp16.
 *   MOE_FMT_E2M1: 4-bit e2m1 codes (the OCP microscaling FP4 element: sign bit
 *                 3, exponent bits 1-2 with bias 1, mantissa bit 0; values 0,
 *                 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives); weight i at bits
 *                 4(i%2) of byte i/2 (low nibble first); a row of K weights =
 *                 K/2 bytes + K/32 fp16.  Its int32 block dots are of TWICE the
 *                 values (exact integers), so the weight scale enters halved.
 *                 (The pages' own low-bit formats are not defined on them; this
 *                 is a 4-bit format GB300's tensor cores take natively.) */
typedef enum { MOE_FMT_Q8_0 = 0, MOE_FMT_Q2S = 1, MOE_FMT_E2M1 = 2 } moe_fmt;

/* One quantised matrix of all experts: q = code plane, scale = fp16 bits.
 * q must be aligned to 32 bytes (MOE_FMT_Q8_0), 8 (MOE_FMT_Q2S) or 16
 * (MOE_FMT_E2M1), scale to 2 (else MOE_ERR_INVALID_ARG).  Every kernel path
 * takes planes whose codes and scales are 16-byte aligned; with less aligned
 * ones the kernels that copy them in 16-byte units (the fused decode kernel,
 * the streamed GEMV for the matrices concerned, the tensor cores) are not
 * used: the same integer block dots, outputs within the layer tolerance. */
typedef struct {
  const void *q;
  const uint16_t *scale;
} moe_mat;

/* Scoring of a router logit l (both with the spec-exp of moe_layer's router):
 * MOE_SCORE_SIGMOID        p = 1/(1+e^-l)          (GLM-5.2 "sigmoid routing
 *                          with top-8" and Hy3's sigmoid router: "256 experts,
 *                          512 lines", section "Why GLM-5.2 in an engine built for
 *                          DeepSeek"; NeutronStar README, Hy3 paragraph)
 * MOE_SCORE_SQRT_SOFTPLUS  p = sqrt(softplus(l)), softplus(l) = max(l,0) +
 *                          log1p(e^-|l|), log1p by the atanh series in
 *                          z = y/(2+y) to z^15 (DeepSeek's scoring with top-6 and
 *                          scale 1.5: "256 experts, 512 lines", section "The
 *                          constant that always said 256").
 * Selection uses c = p + bias; weights w_j = s * p_j / sum_j p_j. */
typedef enum { MOE_SCORE_SIGMOID = 0, MOE_SCORE_SQRT_SOFTPLUS = 1 } moe_score;

/* flags */
/* Write sampled int32 block dots into the workspace (moe_ws_layout.tap_gu /
 * tap_dn) on every path, the fused decode kernel included, from the same dp4a
 * or tensor-core results the outputs are built from; y is unchanged. */
#define MOE_FLAG_DEBUG_TAPS 0x1u
#define MOE_FLAG_FORCE_GEMV 0x2u /* every expert on the dp4a path (no tensor-core path) */
#define MOE_FLAG_FORCE_TC 0x4u   /* every routed expert with >= 1 row on the tensor path */
/* Failure-detection test only: the fused decode kernel never publishes its
 * routing result, so its bounded waits run out (~10 ms) and the call's error
 * word reports MOE_ERR_TIMEOUT; nothing faults and the context stays usable. */
#define MOE_FLAG_TEST_STALL 0x8u
/* Tracing: the fused decode kernel writes 32 uint64 per CTA (timestamps and
 * cycle counts of its waits and phases) into the workspace's trace region. */
#define MOE_FLAG_TRACE 0x10u

typedef struct {
  uint32_t n_expert; /* E, 1..1024 */
  uint32_t top_k;    /* k, 1..E (and <= 32) */
  uint32_t d;        /* hidden size, multiple of 32 */
  uint32_t f;        /* routed expert width, multiple of 32 */
  uint32_t f_shared; /* shared expert width, multiple of 32; 0 = no shared expert */
  int32_t routed_fmt;/* moe_fmt of the routed experts (the shared expert is Q8_0) */
  float s;           /* routing scale */
  uint32_t flags;    /* MOE_FLAG_* */
  uint32_t score;    /* moe_score: how a logit becomes the expert's score */
} moe_desc;

/* Routed experts, expert-major: gate, up [E][f][d]; down [E][d][f] (codes; for
 * Q2S the last dimension is in bytes = K/4), scales [E][rows][K/32].
 * Shared expert (Q8_0): s_gate, s_up [f_shared][d]; s_down [d][f_shared].
 *
 * Optional expert -> slot indirection, for routed experts cached in HBM from a
 * host tier (moe_cache_*): expert_slot (device int32 [E], 4-byte aligned, caller-
 * owned) gives the slot whose weights expert e uses, and gate/up/down then hold
 * n_slots expert-sized slots ([n_slots][f][d], ...) instead of E experts.
 * expert_slot == NULL: slot = expert, n_slots is ignored.  Every expert a call
 * selects must map to a slot in [0, n_slots): one that does not fails the call's
 * device check (MOE_ERR_DEVICE_CHECK via moe_check_device_error) before any of
 * its weights are read; the entries of unselected experts are not read. */
typedef struct {
  moe_mat gate, up, down;
  moe_mat s_gate, s_up, s_down;
  const int32_t *expert_slot;
  uint32_t n_slots;
} moe_weights;

/* The first MOE_WS_FIXED_BYTES of every workspace have a fixed layout: the
 * device error word at offset 0 and, from offset 256, MOE_SYNC_BYTES of
 * counters used by the fused decode kernel and by the streamed GEMV's chunk
 * queues (words 2048..2051).  A workspace must be zero-filled
 * once after it is allocated; every call that completes leaves the counters
 * ready for the next (most zeroed again, two counting calls), so one workspace
 * can serve calls of any desc and T.  A call whose waits timed out may leave
 * them mid-count: moe_check_device_error, reporting MOE_ERR_TIMEOUT, zeroes
 * the whole fixed head, after which the workspace serves calls again.  Every
 * byte past the fixed head is written by a call before that call reads it. */
#define MOE_SYNC_BYTES ((size_t)16384)
#define MOE_WS_FIXED_BYTES ((size_t)256 + MOE_SYNC_BYTES)

/* Regions of the workspace (byte offsets), for debug taps and tests.
 * Rows of the expert FFN are "slots": routed rows at p = pos[t*k+j] in [0, R),
 * shared rows at R + t, R = T*k.  Widths use fmax = max(f, f_shared). */
typedef struct {
  size_t idx, w, off, perm, pos; /* moe_layer's routing results */
  size_t xq, xs;                 /* int8 [T][d], fp32 [T][d/32] */
  size_t hq, hs;                 /* int8 [R+T][fmax], fp32 [R+T][fmax/32] */
  size_t h, o;                   /* fp32 [R+T][fmax], fp32 [R+T][d] */
  size_t plan;                   /* internal work list */
  size_t sync;                   /* counters of the fused decode kernel and the streamed
                                    GEMV's chunk queues (offset 256) */
  size_t tap_gu, tap_dn;         /* int32 taps (MOE_FLAG_DEBUG_TAPS) */
  size_t trace;                  /* uint64 [1024][32] (MOE_FLAG_TRACE) */
  size_t xperm, xsperm, hperm;   /* tensor-core path: fp16 x codes [R+T][d], fp32 x scales
                                    [R+T][d/32], fp16 h codes [R+T][fmax], in slot order */
  size_t xt, ht;                 /* 2-bit routed weights: int8 x codes [T][d] and h codes
                                    [R+T][fmax] with each 16-code group stored 4x4
                                    transposed (byte 4i+j = code 4j+i); 0 otherwise */
  size_t rseg;                   /* router partial sums fp32 [T][E][ceil(d/1024)] of the
                                    fused decode path (T <= 2); 0 otherwise */
  size_t lidx, lw;               /* moe_stream_layer's lookahead picks [T][k] int32, fp32 */
  size_t err;                    /* uint32 device error word: always offset 0 */
  size_t total;
  uint32_t n_tap;                /* tapped features per row (gate/up and down) */
} moe_ws_layout;

/* Tap layout: gate/up: tap_gu[slot][2][n_tap][d/32] int32 (0 = gate, 1 = up) for
 * the features n_j = (j * width / n_tap + j) % width, j < n_tap;
 * down: tap_dn[slot][n_tap][fmax/32] int32 for outputs m_j = (j * d / n_tap + j) % d. */

/* Workspace bytes moe_ffn / moe_layer need for T tokens (0 on invalid desc). */
size_t moe_workspace_size(const moe_desc *desc, uint32_t T);
moe_status moe_workspace_layout(const moe_desc *desc, uint32_t T, moe_ws_layout *out);

/* Router + permutation.  logits [T][E], bias [E] (fp32) -> idx [T][k] int32,
 * w [T][k] fp32, off [E+1] int32, perm [T*k] int32, pos [T*k] int32.
 * Needs no workspace (ws may be NULL). T = 0 writes off = 0 and returns MOE_OK. */
moe_status moe_route(const moe_desc *desc, const float *logits, const float *bias, uint32_t T,
                     int32_t *idx, float *w, int32_t *off, int32_t *perm, int32_t *pos,
                     void *ws, size_t ws_bytes, void *stream);

/* Expert FFN + shared expert + combine for routing results produced by
 * moe_route (or any equivalent producer): x [T][d] fp32 -> y [T][d] fp32. */
moe_status moe_ffn(const moe_desc *desc, const moe_weights *wts, const float *x, uint32_t T,
                   const int32_t *idx, const float *w, const int32_t *off,
                   const int32_t *perm, const int32_t *pos, float *y, void *ws,
                   size_t ws_bytes, void *stream);

/* The whole layer: moe_route into the workspace, then moe_ffn. */
moe_status moe_layer(const moe_desc *desc, const moe_weights *wts, const float *x,
                     const float *logits, const float *bias, uint32_t T, float *y, void *ws,
                     size_t ws_bytes, void *stream);

/* moe_layer with timing markers for profiling.  `events` holds n_events
 * cudaEvent_t handles (created by the caller); events[0] is recorded on
 * `stream` before the first stage and events[i] after stage i-1, for
 * i < n_events (as external records, so they also work inside CUDA graph
 * capture).  Stage names come from moe_stage_name.  events == NULL or
 * n_events == 0 makes this identical to moe_layer. */
moe_status moe_layer_timed(const moe_desc *desc, const moe_weights *wts, const float *x,
                           const float *logits, const float *bias, uint32_t T, float *y,
                           void *ws, size_t ws_bytes, void *stream, void *const *events,
                           uint32_t n_events);

/* Router logits in front of the scoring: logits[t][e] = sum_i x[t][i] *
 * w_router[e][i] in fp32 in one fixed order -- the inputs form segments of
 * 1024; in each, lane l (of 32) accumulates i = l, l+32, ... ascending with
 * fused multiply-adds, the 32 partial sums are combined pairwise over lane
 * distances 16, 8, 4, 2, 1, and the segment totals are added in ascending
 * order -- so that any implementation of that order gets the same bits (the
 * expert picks downstream depend on them).  The pages give no precision for the router GEMM; fp32
 * weights and this order are this library's definition.
 * x: [T][d] fp32, w_router: [E][d] fp32, logits: [T][E] fp32, all device
 * pointers (caller-owned, 16-byte aligned).  Asynchronous on `stream`;
 * MOE_ERR_INVALID_ARG on a bad desc, d > 32768, or a NULL pointer with T > 0. */
moe_status moe_router_logits(const moe_desc *desc, const float *w_router, const float *x,
                             uint32_t T, float *logits, void *stream);

/* The layer from the hidden state: the router logits of moe_router_logits
 * (same order, same bits), written to `logits` [T][E] fp32 (an output here,
 * caller-owned), then moe_layer on them -- the router front end fused in front
 * of the scoring and top-k ("256 experts, 512 lines", "The constant that
 * always said 256": per token, n_expert logits feed the expert scores).
 * On the fused decode path (moe_layer_path "fused_decode", T <= 2) the logits
 * are computed inside the decode kernel: every CTA takes a share of the
 * (expert, 1024-input segment) partial sums, writes them to the workspace
 * (moe_ws_layout.rseg), and every CTA then adds each logit's segments in
 * ascending order itself, while the shared expert's weights already stream.
 * On the multi-kernel path the moe_router_logits kernel runs first.
 * w_router [E][d] fp32 and x 16-byte aligned; d <= 32768; otherwise as
 * moe_layer (workspace from moe_workspace_size, MOE_ERR_INVALID_ARG on a bad
 * argument before anything is launched). */
moe_status moe_layer_from_x(const moe_desc *desc, const moe_weights *wts,
                            const float *w_router, const float *x, const float *bias, uint32_t T,
                            float *logits, float *y, void *ws, size_t ws_bytes, void *stream);

/* ---- Expert-parallel split ----
 * The layer restricted to one rank's share of the experts: routing over all
 * n_expert as in moe_layer (every rank routes every token the same way), then
 *   y[t] = [with_shared] o_shared[t] + sum over slots j with
 *          expert_begin <= idx[t][j] < expert_end of w[t][j] * o[t][j]
 * (shared first, then the owned slots in slot order).  Ranks whose ranges
 * partition [0, n_expert), with with_shared set on exactly one of them, give
 * partial outputs whose sum is the layer (a sum all-reduce of y: the
 * expert-parallel residency the pages name as the next multi-GPU lever,
 * NeutronStar README, next-levers paragraph, and the two-worker split of
 * NeutronStar glm-local README, "Roadmap"); the sum's fp32 order differs from
 * moe_layer's, so it matches within the output tolerance, not bit for bit.
 * Only the owned experts' weights are read: with moe_weights.expert_slot a
 * rank holds its own experts only (the slots of unowned experts are never
 * read, and need not be valid).  Workspace as moe_layer.  An empty range
 * (expert_begin == expert_end) computes the shared expert alone (or y = 0).
 * MOE_ERR_INVALID_ARG unless expert_begin <= expert_end <= n_expert. */
moe_status moe_layer_experts(const moe_desc *desc, const moe_weights *wts, const float *x,
                             const float *logits, const float *bias, uint32_t T,
                             uint32_t expert_begin, uint32_t expert_end, int32_t with_shared,
                             float *y, void *ws, size_t ws_bytes, void *stream);

/* moe_ffn restricted the same way: the expert FFN and combine of the owned
 * experts (and the shared expert if with_shared) for routing results computed
 * elsewhere -- the compute step of an all-to-all dispatch, where a rank receives
 * the rows (x and their full routing) that name at least one of its experts. */
moe_status moe_ffn_experts(const moe_desc *desc, const moe_weights *wts, const float *x,
                           uint32_t T, const int32_t *idx, const float *w, const int32_t *off,
                           const int32_t *perm, const int32_t *pos, uint32_t expert_begin,
                           uint32_t expert_end, int32_t with_shared, float *y, void *ws,
                           size_t ws_bytes, void *stream);

/* Which implementation moe_layer uses for (desc, T) on the current device:
 * "fused_decode" (one persistent kernel, T <= 2) or "multi_kernel".  The fused
 * kernel reads x in 16-byte vectors, so a call whose x (or a weight plane, see
 * moe_mat) is not 16-byte aligned takes the multi-kernel path whatever this
 * returns (x and y need only the 4-byte alignment of their floats). */
const char *moe_layer_path(const moe_desc *desc, uint32_t T);

/* Row threshold of the tensor-core path of moe_layer for (desc, T) on the
 * current device (6 for Q8_0 and Q2S routed weights, 4 for E2M1, 0 with
 * MOE_FLAG_FORCE_TC): an expert (the shared expert included, with T rows, when
 * f_shared == f) whose routed row count exceeds it runs its block dots on
 * tcgen05 tensor cores, the rest on the dp4a GEMV -- provided those experts'
 * gate/up tiles (128 features x 64 rows each) number at least the device's SM
 * count; with fewer, every expert of the call runs on the GEMV (a nearly empty
 * tensor kernel would leave most SMs idle).  MOE_FLAG_FORCE_TC sends every
 * expert to the tensor cores.  2-bit routed weights take the same path: their
 * codes are decoded to fp16 (2c - 3, exact) on the way to the MMA.  -1 when no
 * expert of such a call can take the tensor path (the fused decode path, dims
 * not a multiple of 256, MOE_FLAG_FORCE_GEMV, fewer than 32 tokens without
 * MOE_FLAG_FORCE_TC, or T at most the threshold). */
int32_t moe_tc_min_rows(const moe_desc *desc, uint32_t T);

/* Name of stage i of that path (what moe_layer_timed's events bracket),
 * NULL past the last stage. */
const char *moe_layer_stage_name(const moe_desc *desc, uint32_t T, uint32_t i);

/* ---- Host-tier expert streaming: an HBM expert cache over host memory ----
 * The pages stream routed experts per token from a slower tier into a GPU-side
 * expert cache, keep the hottest experts in an LFU cache, load the union of a
 * batch's experts once, and prefetch the next layer's experts by running its
 * router early (NeutronStar glm-local README, "SSD streaming optimizations":
 * the host expert cache with LFU eviction and the cross-layer router-lookahead
 * prefetch; "Long-prompt prefill": one union read serves a chunk).  Here the
 * slow tier is host memory (pinned; on GB300 the Grace LPDDR across NVLink-C2C)
 * holding every layer's routed experts, and the cache is an arena of n_slots
 * expert-sized slots in HBM shared by all layers; moe_weights.expert_slot
 * points the layer kernels at the slots.
 *
 * Policy (deterministic): each moe_cache_ensure call counts one lookup for every
 * distinct expert it names (the LFU frequency, kept while the expert is evicted)
 * and stamps it as the most recent use.  A missing expert takes the lowest free
 * slot, else evicts the resident expert with the fewest lookups, ties to the
 * least recent use, then to the lower (layer, expert).  Never evicted: the
 * experts of the call itself and, for a prefetch, those of the latest ensure
 * (their layer may still be running).  A call whose union exceeds what it may
 * evict fails with MOE_ERR_WORKSPACE before copying anything.
 * Ordering: ensure copies on its stream (the compute stream), so they follow
 * every kernel enqueued there before; prefetch copies on their own stream start
 * after the latest ensure's copies (which go first on the link, and follow every
 * earlier use of an evicted slot), and an ensure that needs a prefetched expert
 * makes its stream wait for that copy. */
typedef struct moe_cache moe_cache;

typedef struct {
  uint64_t lookups;        /* distinct experts named by moe_cache_ensure calls */
  uint64_t hits;           /* ... already resident (loaded before, or prefetched) */
  uint64_t misses;         /* ... loaded by the ensure call itself */
  uint64_t prefetch_loads; /* experts loaded by moe_cache_prefetch */
  uint64_t prefetch_hits;  /* prefetched experts later named by an ensure while resident */
  uint64_t evictions;
  uint64_t bytes_h2d;      /* weight bytes copied host -> HBM */
} moe_cache_stats;

#define MOE_CACHE_POLICY_ONLY 1u /* no device work: moe_cache_plan only (tests, planning) */

/* host_layers[n_layers]: each layer's routed gate/up/down planes in pinned host
 * memory, expert-major as in moe_weights (shared-expert fields and expert_slot
 * ignored).  arena: gate/up/down planes of n_slots expert slots in device memory
 * (same per-expert layout).  slot_table: device int32 [n_layers][E], written by
 * the cache (layer l's moe_weights.expert_slot = slot_table + l*E).  All memory
 * is caller-owned and must outlive the cache; the cache itself allocates host
 * memory and CUDA events only.  MOE_ERR_INVALID_ARG on a bad argument. */
moe_status moe_cache_create(const moe_desc *desc, uint32_t n_layers,
                            const moe_weights *host_layers, const moe_weights *arena,
                            uint32_t n_slots, int32_t *slot_table, uint32_t flags,
                            moe_cache **out);
void moe_cache_destroy(moe_cache *cache);

/* Make the distinct experts of experts[0..n) of `layer` resident, copying
 * misses host -> HBM on `stream`, and upload the layer's slot table on `stream`.
 * Experts outside [0, E) are MOE_ERR_INVALID_ARG. */
moe_status moe_cache_ensure(moe_cache *cache, uint32_t layer, const int32_t *experts,
                            uint32_t n, void *stream);

/* Load what of experts[0..n) of `layer` is missing on `stream` (a side stream),
 * without counting lookups; stops quietly when nothing may be evicted. */
moe_status moe_cache_prefetch(moe_cache *cache, uint32_t layer, const int32_t *experts,
                              uint32_t n, void *stream);

/* The policy step of ensure (prefetch != 0: of prefetch) with no device work:
 * updates the cache state as the call would and reports the experts it would
 * load, their slots and the (layer*E + expert) each evicts (-1: a free slot);
 * the arrays hold n entries, n_loaded receives the count. */
moe_status moe_cache_plan(moe_cache *cache, uint32_t layer, const int32_t *experts, uint32_t n,
                          int prefetch, int32_t *loaded, int32_t *slots, int64_t *evicted,
                          uint32_t *n_loaded);

/* Layers the cache was created for (0 for NULL). */
uint32_t moe_cache_layers(const moe_cache *cache);

/* Slot of (layer, expert), -1 when not resident or out of range. */
int32_t moe_cache_slot(const moe_cache *cache, uint32_t layer, int32_t expert);
moe_status moe_cache_get_stats(const moe_cache *cache, moe_cache_stats *out);

/* One decode/prefill step of one layer with its routed experts served by the
 * cache: route x's logits on the device, read the picks back (the stream is
 * synchronised once), make their union resident (moe_cache_ensure on `stream`),
 * then moe_layer on the slot weights.  wts: the layer's shared-expert planes
 * (routed fields and expert_slot ignored: the arena and the layer's slot table
 * are used).  next_logits / next_bias (optional, device, [T][E] / [E]): the next
 * layer's router applied early to this layer's x -- their top-k picks are
 * read back with this layer's and prefetched for layer + 1 on prefetch_stream
 * while this layer runs.  Workspace as moe_layer.  A call with more routed rows
 * than any before on this cache first grows the cache's pinned read-back
 * buffer (MOE_ERR_CUDA if that allocation fails). */
moe_status moe_stream_layer(moe_cache *cache, uint32_t layer, const moe_desc *desc,
                            const moe_weights *wts, const float *x, const float *logits,
                            const float *bias, uint32_t T, const float *next_logits,
                            const float *next_bias, float *y, void *ws, size_t ws_bytes,
                            void *stream, void *prefetch_stream);

/* ---- Allocation-free variant (the pages have no counterpart of this) ----
 * moe_layer without a workspace argument, for callers that cannot allocate
 * device memory: code running inside an engine whose device-memory arena was
 * reserved up front, plugins and plain-C hosts without an allocator, and
 * latency-critical paths that must not touch the allocator.  The scratch the
 * layer needs lives in one static device array of MOE_NOALLOC_SCRATCH_BYTES,
 * held by every GPU that loads the library until the process exits.
 * - Calls whose moe_workspace_size(desc, T) exceeds it return
 *   MOE_ERR_WORKSPACE (moe_last_error says why) and launch nothing.  For the
 *   E=256 / d=6144 / f=2048 layer with a shared expert that is T <= 32.
 * - All calls on a device share the array, which keeps the last call's
 *   contents; what must start at zero (error word, counters) is zero-filled
 *   at set-up and the counters are left zeroed by every call that completes.
 *   The device error word (bad weight slots, timed-out waits) keeps its bits
 *   until moe_check_device_error(NULL, 0, stream) reads and clears it; after a
 *   timeout that call also zeroes the counters.  Calls that overlap on the GPU
 *   race on the array: serialise them.
 * - The first call on each device looks up the array's device address,
 *   caches it and zero-fills the array's head on that call's stream; make
 *   that first call before any stream capture begins.
 * - Allocates nothing (no cudaMalloc/cudaFree or allocating library call).
 * Inputs and outputs are the caller's device buffers, as for moe_layer. */
#define MOE_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
moe_status moe_layer_noalloc(const moe_desc *desc, const moe_weights *wts, const float *x,
                             const float *logits, const float *bias, uint32_t T, float *y,
                             void *stream);

/* Synchronise `stream` and read (then clear) the workspace's device error word
 * (the first 4 bytes of any workspace), which holds every bit the calls on that
 * workspace set since it was last cleared.  MOE_OK if no kernel flagged a
 * fault; MOE_ERR_TIMEOUT if a bounded wait gave up (the whole fixed head, the
 * counters included, is then zeroed: ws_bytes >= MOE_WS_FIXED_BYTES);
 * MOE_ERR_DEVICE_CHECK for bad routing inputs or weight slots.
 * ws == NULL with ws_bytes == 0: the same for moe_layer_noalloc's static
 * scratch on the current device (MOE_OK, with no CUDA call, before the first
 * moe_layer_noalloc call there).  ws == NULL with ws_bytes != 0, or
 * ws_bytes < 4: MOE_ERR_INVALID_ARG. */
moe_status moe_check_device_error(void *ws, size_t ws_bytes, void *stream);

const char *moe_status_string(moe_status st);

/* Name of the CUDA error behind the calling thread's last MOE_ERR_CUDA
 * ("no error" if there was none).  Static storage; do not free. */
const char *moe_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
