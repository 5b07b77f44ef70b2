// moe_api.cu -- the C ABI (moe.h): argument checks, workspace layout and the
// launch sequence.  The host only validates and enqueues; every step of the
// layer runs in this library's kernels on the caller's stream.
#include <string.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

bool desc_ok(const moe_desc *d) {
  if (!d) return false;
  if (d->n_expert < 1 || d->n_expert > 1024) return false;
  if (d->top_k < 1 || d->top_k > d->n_expert || d->top_k > 32) return false;
  if (d->d == 0 || d->d % 32 || d->f == 0 || d->f % 32 || d->f_shared % 32) return false;
  if (d->routed_fmt != MOE_FMT_Q8_0 && d->routed_fmt != MOE_FMT_Q2S &&
      d->routed_fmt != MOE_FMT_E2M1)
    return false;
  if (!(d->s == d->s)) return false;  // NaN scale
  if (d->score != MOE_SCORE_SIGMOID && d->score != MOE_SCORE_SQRT_SOFTPLUS) return false;
  // int32 indexing of rows and work items
  if ((uint64_t)d->n_expert * d->f > (1u << 30) || (uint64_t)d->n_expert * d->d > (1u << 30))
    return false;
  return true;
}

bool mat_ok(const moe_mat &m, int fmt) {
  if (!m.q || !m.scale) return false;
  if (!aligned(m.q, fmt == MOE_FMT_Q2S ? 8 : fmt == MOE_FMT_E2M1 ? 16 : 32)) return false;
  if (!aligned(m.scale, 2)) return false;
  return true;
}

// The fused kernel streams weight rows and their scales with bulk copies, which
// start on 16-byte boundaries: planes that are not 16-byte aligned (moe_mat
// allows less) keep a call on the multi-kernel path.
bool fused_weights_aligned(const moe_desc &d, const moe_weights &w) {
  bool ok = aligned(w.gate.q, 16) && aligned(w.up.q, 16) && aligned(w.down.q, 16) &&
            aligned(w.gate.scale, 16) && aligned(w.up.scale, 16) && aligned(w.down.scale, 16);
  if (d.f_shared)
    ok = ok && aligned(w.s_gate.q, 16) && aligned(w.s_up.q, 16) && aligned(w.s_down.q, 16) &&
         aligned(w.s_gate.scale, 16) && aligned(w.s_up.scale, 16) && aligned(w.s_down.scale, 16);
  return ok;
}

bool weights_ok(const moe_desc *d, const moe_weights *w) {
  if (!w) return false;
  const int f = d->routed_fmt;
  if (!mat_ok(w->gate, f) || !mat_ok(w->up, f) || !mat_ok(w->down, f)) return false;
  if (w->expert_slot) {
    if (!aligned(w->expert_slot, 4) || w->n_slots < 1) return false;
    if ((uint64_t)w->n_slots * d->f > (1u << 30) || (uint64_t)w->n_slots * d->d > (1u << 30))
      return false;
  }
  if (d->f_shared) {
    if (!mat_ok(w->s_gate, MOE_FMT_Q8_0) || !mat_ok(w->s_up, MOE_FMT_Q8_0) ||
        !mat_ok(w->s_down, MOE_FMT_Q8_0))
      return false;
  }
  return true;
}

moe_ws_layout make_layout(const moe_desc *d, uint32_t T) {
  moe_ws_layout L;
  memset(&L, 0, sizeof L);
  const size_t R = (size_t)T * d->top_k;
  const size_t slots = R + (d->f_shared ? T : 0);
  const size_t fmax = d->f > d->f_shared ? d->f : d->f_shared;
  size_t p = 0;
  L.err = p;
  L.sync = 256;
  p = align_up(MOE_WS_FIXED_BYTES);
  L.idx = p; p = align_up(p + R * 4);
  L.w = p; p = align_up(p + R * 4);
  L.off = p; p = align_up(p + (size_t)(d->n_expert + 1) * 4);
  L.perm = p; p = align_up(p + R * 4);
  L.pos = p; p = align_up(p + R * 4);
  L.plan = p; p = align_up(p + PlanView::ints(d->n_expert) * 4);
  L.xq = p; p = align_up(p + (size_t)T * d->d);
  L.xs = p; p = align_up(p + (size_t)T * (d->d / 32) * 4);
  L.h = p; p = align_up(p + slots * fmax * 4);
  L.hq = p; p = align_up(p + slots * fmax);
  L.hs = p; p = align_up(p + slots * (fmax / 32) * 4);
  L.o = p; p = align_up(p + slots * d->d * 4);
  L.n_tap = kNTap;
  if (d->flags & MOE_FLAG_DEBUG_TAPS) {
    L.tap_gu = p; p = align_up(p + slots * 2 * kNTap * (d->d / 32) * 4);
    L.tap_dn = p; p = align_up(p + slots * kNTap * (fmax / 32) * 4);
  } else {
    L.tap_gu = L.tap_dn = 0;
  }
  L.xperm = L.xsperm = L.hperm = 0;
  if (tc_possible(*d, T)) {
    L.xperm = p; p = align_up(p + slots * d->d * 2);
    L.xsperm = p; p = align_up(p + slots * (d->d / 32) * 4);
    L.hperm = p; p = align_up(p + slots * fmax * 2);
  }
  L.xt = L.ht = 0;
  if (d->routed_fmt == MOE_FMT_Q2S) {
    L.xt = p; p = align_up(p + (size_t)T * d->d);
    L.ht = p; p = align_up(p + slots * fmax);
  }
  L.rseg = 0;
  if (T >= 1 && T <= 2) {
    L.rseg = p; p = align_up(p + (size_t)T * d->n_expert * ((d->d + kRouterSeg - 1) / kRouterSeg) * 4);
  }
  L.lidx = p; p = align_up(p + R * 4);
  L.lw = p; p = align_up(p + R * 4);
  L.trace = 0;
  if (d->flags & MOE_FLAG_TRACE) {
    L.trace = p; p = align_up(p + (size_t)1024 * 32 * 8);
  }
  L.total = p;
  return L;
}

int sm_count_of_current_device() {
  int dev = 0, n = kSmCount;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : kSmCount;
}

thread_local const char *t_last_error = "no error";

moe_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  t_last_error = cudaGetErrorName(e);
  return MOE_ERR_CUDA;
}

Ctx make_ctx(const moe_desc *d, const moe_weights *w, uint32_t T, void *ws, void *stream) {
  Ctx c;
  memset(&c, 0, sizeof c);
  c.desc = *d;
  if (w) c.wts = *w;
  c.T = T;
  c.R = T * d->top_k;
  c.fmax = d->f > d->f_shared ? d->f : d->f_shared;
  c.wexp = (w && w->expert_slot) ? w->n_slots : d->n_expert;
  c.ws = (uint8_t *)ws;
  c.L = make_layout(d, T);
  c.stream = (cudaStream_t)stream;
  c.sm_count = sm_count_of_current_device();
  c.e_lo = 0;
  c.e_hi = d->n_expert;
  c.shared_on = true;
  c.chained = false;
  return c;
}

const char *const kStageNames[] = {"route",   "permute",   "plan", "quant_x", "tc_prepare",
                                   "gateup",  "requant",   "gateup_tc", "down", "down_tc",
                                   "combine"};
constexpr uint32_t kNumStages = sizeof(kStageNames) / sizeof(kStageNames[0]);
const char *const kFusedStageNames[] = {"decode_fused"};
constexpr uint32_t kNumFusedStages = 1;

// optional timing markers: events[i] after stage i-1
struct Marks {
  void *const *ev;
  uint32_t n;
  cudaStream_t s;
  bool capturing;
  Marks(void *const *e, uint32_t k, cudaStream_t st) : ev(e), n(k), s(st), capturing(false) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (ev && n && cudaStreamIsCapturing(s, &cs) == cudaSuccess)
      capturing = cs == cudaStreamCaptureStatusActive;
  }
  cudaError_t mark(uint32_t i) const {
    if (!ev || i >= n) return cudaSuccess;
    // inside stream capture an external record becomes an event-record node
    return capturing ? cudaEventRecordWithFlags((cudaEvent_t)ev[i], s, cudaEventRecordExternal)
                     : cudaEventRecord((cudaEvent_t)ev[i], s);
  }
};

// FFN stages shared by moe_ffn and moe_layer (stage numbers 2..10)
moe_status run_ffn(const Ctx &c, const float *x, const int32_t *idx, const float *w,
                   const int32_t *off, const int32_t *perm, const int32_t *pos, float *y,
                   const Marks &mk) {
  uint32_t *err = (uint32_t *)(c.ws + c.L.err);
  cudaError_t e;
  if ((e = launch_plan(c, off, idx, perm, pos, err)) != cudaSuccess) return from_cuda(e);
  if ((e = mk.mark(3)) != cudaSuccess) return from_cuda(e);
  if ((e = launch_quant_x(c, x)) != cudaSuccess) return from_cuda(e);
  if ((e = mk.mark(4)) != cudaSuccess) return from_cuda(e);
  // tensor-core experts possible for this desc and T
  const bool tc = c.L.xperm != 0 && tc_supported(c.desc) && tc_weights_aligned(c);
  if (tc && (e = launch_tc_prepare(c, perm)) != cudaSuccess) return from_cuda(e);
  if ((e = mk.mark(5)) != cudaSuccess) return from_cuda(e);
  if ((e = launch_gateup(c, perm)) != cudaSuccess) return from_cuda(e);
  if ((e = mk.mark(6)) != cudaSuccess) return from_cuda(e);
  // requantises h of every slot; the tensor path then writes its own slots' codes
  if ((e = launch_requant_h(c)) != cudaSuccess) return from_cuda(e);
  if ((e = mk.mark(7)) != cudaSuccess) return from_cuda(e);
  if (tc && (e = launch_tc(c, 2)) != cudaSuccess) return from_cuda(e);
  if ((e = mk.mark(8)) != cudaSuccess) return from_cuda(e);
  if ((e = launch_down(c)) != cudaSuccess) return from_cuda(e);
  if ((e = mk.mark(9)) != cudaSuccess) return from_cuda(e);
  if (tc && (e = launch_tc(c, 1)) != cudaSuccess) return from_cuda(e);
  if ((e = mk.mark(10)) != cudaSuccess) return from_cuda(e);
  if ((e = launch_combine(c, w, pos, idx, y)) != cudaSuccess) return from_cuda(e);
  if ((e = mk.mark(11)) != cudaSuccess) return from_cuda(e);
  return MOE_OK;
}

// w_router non-null: the router logits are computed from x into `logits`
// (an output then); else `logits` is the caller's input
// e_lo, e_hi, shared_on: the routed experts [e_lo, e_hi) and the shared expert
// (if shared_on) are the ones computed; e_hi == 0 means all experts
moe_status run_layer(const moe_desc *desc, const moe_weights *wts, const float *x,
                     const float *logits, const float *bias, uint32_t T, float *y, void *ws,
                     size_t ws_bytes, void *stream, void *const *events, uint32_t n_events,
                     const float *w_router = nullptr, uint32_t e_lo = 0, uint32_t e_hi = 0,
                     bool shared_on = true, bool no_routed = false) {
  if (!desc_ok(desc) || !weights_ok(desc, wts)) return MOE_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !logits || !bias || !y)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && w_router &&
      (!aligned(w_router, 16) || !aligned(x, 16) || !aligned(logits, 4) || desc->d > 32768 ||
       (uint64_t)T * desc->n_expert > 0x7fffffffull))
    return MOE_ERR_INVALID_ARG;
  if ((uint64_t)T * desc->top_k > (1u << 30)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < make_layout(desc, T).total) return MOE_ERR_WORKSPACE;
  Ctx c = make_ctx(desc, wts, T, ws, stream);
  if (e_hi) {
    c.e_lo = e_lo;
    c.e_hi = e_hi;
  }
  if (no_routed) c.e_lo = c.e_hi = 0;  // an empty range: the shared expert alone
  c.shared_on = shared_on;
  Marks mk(events, n_events, c.stream);
  int32_t *idx = (int32_t *)(c.ws + c.L.idx);
  float *w = (float *)(c.ws + c.L.w);
  int32_t *off = (int32_t *)(c.ws + c.L.off);
  int32_t *perm = (int32_t *)(c.ws + c.L.perm);
  int32_t *pos = (int32_t *)(c.ws + c.L.pos);
  uint32_t *err = (uint32_t *)(c.ws + c.L.err);
  cudaError_t e;
  float *logits_out = const_cast<float *>(w_router ? logits : nullptr);
  // the fused kernel reads x in 16-byte vectors and copies weight planes in
  // 16-byte units: an x or planes not 16-byte aligned take the multi-kernel
  // path (whose quantiser reads x either way)
  if (T > 0 && fused_eligible(c) && aligned(x, 16) && fused_weights_aligned(*desc, *wts)) {
    if ((e = mk.mark(0)) != cudaSuccess) return from_cuda(e);
    if ((e = launch_decode_fused(c, x, logits, bias, y, w_router, logits_out)) != cudaSuccess)
      return from_cuda(e);
    if ((e = mk.mark(1)) != cudaSuccess) return from_cuda(e);
    return MOE_OK;
  }
  if ((e = mk.mark(0)) != cudaSuccess) return from_cuda(e);
  if (w_router && T > 0 &&
      (e = launch_router_logits(c.desc, w_router, x, T, logits_out, c.stream)) != cudaSuccess)
    return from_cuda(e);
  if (w_router && T > 0) c.chained = true;  // the router kernel is on the stream
  if ((e = launch_route(c, logits, bias, idx, w)) != cudaSuccess) return from_cuda(e);
  if ((e = mk.mark(1)) != cudaSuccess) return from_cuda(e);
  if ((e = launch_permute(c, idx, off, perm, pos, err)) != cudaSuccess) return from_cuda(e);
  if ((e = mk.mark(2)) != cudaSuccess) return from_cuda(e);
  return run_ffn(c, x, idx, w, off, perm, pos, y, mk);
}

}  // namespace

// Entry points for other translation units of the library.
moe_status layer_on_workspace(const moe_desc *desc, const moe_weights *wts, const float *x,
                              const float *logits, const float *bias, uint32_t T, float *y,
                              void *ws, size_t ws_bytes, void *stream) {
  return run_layer(desc, wts, x, logits, bias, T, y, ws, ws_bytes, stream, nullptr, 0);
}

void set_last_error(const char *msg) { t_last_error = msg; }

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_size(const moe_desc *desc, uint32_t T) {
  if (!desc_ok(desc)) return 0;
  return make_layout(desc, T).total;
}

moe_status moe_workspace_layout(const moe_desc *desc, uint32_t T, moe_ws_layout *out) {
  if (!desc_ok(desc) || !out) return MOE_ERR_INVALID_ARG;
  *out = make_layout(desc, T);
  return MOE_OK;
}

moe_status moe_route(const moe_desc *desc, const float *logits, const float *bias, uint32_t T,
                     int32_t *idx, float *w, int32_t *off, int32_t *perm, int32_t *pos,
                     void *ws, size_t ws_bytes, void *stream) {
  (void)ws;
  (void)ws_bytes;
  if (!desc_ok(desc)) return MOE_ERR_INVALID_ARG;
  if (!off) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !bias || !idx || !w || !perm || !pos)) return MOE_ERR_INVALID_ARG;
  if ((uint64_t)T * desc->top_k > (1u << 30)) return MOE_ERR_INVALID_ARG;
  Ctx c = make_ctx(desc, nullptr, T, nullptr, stream);
  cudaError_t e;
  if ((e = launch_route(c, logits, bias, idx, w)) != cudaSuccess) return from_cuda(e);
  // moe_route's own idx is always in range, so the device error word is not needed
  if ((e = launch_permute(c, idx, off, perm, pos, nullptr)) != cudaSuccess) return from_cuda(e);
  return MOE_OK;
}

moe_status moe_ffn(const moe_desc *desc, const moe_weights *wts, const float *x, uint32_t T,
                   const int32_t *idx, const float *w, const int32_t *off,
                   const int32_t *perm, const int32_t *pos, float *y, void *ws,
                   size_t ws_bytes, void *stream) {
  if (!desc_ok(desc) || !weights_ok(desc, wts)) return MOE_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign) || !off) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !idx || !w || !perm || !pos || !y)) return MOE_ERR_INVALID_ARG;
  if ((uint64_t)T * desc->top_k > (1u << 30)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < make_layout(desc, T).total) return MOE_ERR_WORKSPACE;
  Ctx c = make_ctx(desc, wts, T, ws, stream);
  return run_ffn(c, x, idx, w, off, perm, pos, y, Marks(nullptr, 0, c.stream));
}

moe_status moe_layer(const moe_desc *desc, const moe_weights *wts, const float *x,
                     const float *logits, const float *bias, uint32_t T, float *y, void *ws,
                     size_t ws_bytes, void *stream) {
  return run_layer(desc, wts, x, logits, bias, T, y, ws, ws_bytes, stream, nullptr, 0);
}

moe_status moe_layer_timed(const moe_desc *desc, const moe_weights *wts, const float *x,
                           const float *logits, const float *bias, uint32_t T, float *y,
                           void *ws, size_t ws_bytes, void *stream, void *const *events,
                           uint32_t n_events) {
  return run_layer(desc, wts, x, logits, bias, T, y, ws, ws_bytes, stream, events, n_events);
}

moe_status moe_layer_experts(const moe_desc *desc, const moe_weights *wts, const float *x,
                             const float *logits, const float *bias, uint32_t T,
                             uint32_t expert_begin, uint32_t expert_end, int32_t with_shared,
                             float *y, void *ws, size_t ws_bytes, void *stream) {
  if (!desc_ok(desc) || expert_begin > expert_end || expert_end > desc->n_expert)
    return MOE_ERR_INVALID_ARG;
  return run_layer(desc, wts, x, logits, bias, T, y, ws, ws_bytes, stream, nullptr, 0, nullptr,
                   expert_begin, expert_end == expert_begin ? 0 : expert_end, with_shared != 0,
                   expert_end == expert_begin);
}

moe_status moe_ffn_experts(const moe_desc *desc, const moe_weights *wts, const float *x,
                           uint32_t T, const int32_t *idx, const float *w, const int32_t *off,
                           const int32_t *perm, const int32_t *pos, uint32_t expert_begin,
                           uint32_t expert_end, int32_t with_shared, float *y, void *ws,
                           size_t ws_bytes, void *stream) {
  if (!desc_ok(desc) || expert_begin > expert_end || expert_end > desc->n_expert)
    return MOE_ERR_INVALID_ARG;
  if (!weights_ok(desc, wts)) return MOE_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign) || !off) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !idx || !w || !perm || !pos || !y)) return MOE_ERR_INVALID_ARG;
  if ((uint64_t)T * desc->top_k > (1u << 30)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < make_layout(desc, T).total) return MOE_ERR_WORKSPACE;
  Ctx c = make_ctx(desc, wts, T, ws, stream);
  c.e_lo = expert_begin;
  c.e_hi = expert_end;
  c.shared_on = with_shared != 0;
  return run_ffn(c, x, idx, w, off, perm, pos, y, Marks(nullptr, 0, c.stream));
}

moe_status moe_layer_from_x(const moe_desc *desc, const moe_weights *wts,
                            const float *w_router, const float *x, const float *bias, uint32_t T,
                            float *logits, float *y, void *ws, size_t ws_bytes, void *stream) {
  if (T > 0 && !w_router) return MOE_ERR_INVALID_ARG;
  return run_layer(desc, wts, x, logits, bias, T, y, ws, ws_bytes, stream, nullptr, 0,
                   T > 0 ? w_router : nullptr);
}

moe_status moe_stream_layer(moe_cache *cache, uint32_t layer, const moe_desc *desc,
                            const moe_weights *wts, const float *x, const float *logits,
                            const float *bias, uint32_t T, const float *next_logits,
                            const float *next_bias, float *y, void *ws, size_t ws_bytes,
                            void *stream, void *prefetch_stream) {
  const moe_desc *cd = cache_desc(cache);
  if (!cd || !desc_ok(desc) || !wts) return MOE_ERR_INVALID_ARG;
  if (cd->n_expert != desc->n_expert || cd->d != desc->d || cd->f != desc->f ||
      cd->routed_fmt != desc->routed_fmt)
    return MOE_ERR_INVALID_ARG;
  if (next_logits && !next_bias) return MOE_ERR_INVALID_ARG;
  moe_weights w = *wts;
  if (!cache_layer_routed(cache, layer, &w)) return MOE_ERR_INVALID_ARG;
  if (!weights_ok(desc, &w)) return MOE_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !logits || !bias || !y)) return MOE_ERR_INVALID_ARG;
  if ((uint64_t)T * desc->top_k > (1u << 30)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < make_layout(desc, T).total) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  Ctx c = make_ctx(desc, &w, T, ws, stream);
  int32_t *idx = (int32_t *)(c.ws + c.L.idx);
  int32_t *lidx = (int32_t *)(c.ws + c.L.lidx);
  const bool look = next_logits != nullptr && layer + 1 < moe_cache_layers(cache);
  const size_t R = c.R;
  int32_t *host = cache_pinned(cache, 2 * R);
  if (!host) {
    set_last_error("moe_stream_layer: cudaHostAlloc failed");
    return MOE_ERR_CUDA;
  }
  // the picks of this layer (and of the next layer's router, run early), read back
  cudaError_t e = launch_route(c, logits, bias, idx, (float *)(c.ws + c.L.w));
  if (e == cudaSuccess && look)
    e = launch_route(c, next_logits, next_bias, lidx, (float *)(c.ws + c.L.lw));
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(host, idx, R * 4, cudaMemcpyDeviceToHost, c.stream);
  if (e == cudaSuccess && look)
    e = cudaMemcpyAsync(host + R, lidx, R * 4, cudaMemcpyDeviceToHost, c.stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c.stream);
  if (e != cudaSuccess) return from_cuda(e);
  moe_status st = moe_cache_ensure(cache, layer, host, (uint32_t)R, stream);
  if (st != MOE_OK) return st;
  if (look) {
    st = moe_cache_prefetch(cache, layer + 1, host + R, (uint32_t)R, prefetch_stream);
    if (st != MOE_OK) return st;
  }
  return run_layer(desc, &w, x, logits, bias, T, y, ws, ws_bytes, stream, nullptr, 0);
}

const char *moe_layer_path(const moe_desc *desc, uint32_t T) {
  if (!desc_ok(desc)) return nullptr;
  Ctx c = make_ctx(desc, nullptr, T, nullptr, nullptr);
  return (T > 0 && fused_eligible(c)) ? "fused_decode" : "multi_kernel";
}

int32_t moe_tc_min_rows(const moe_desc *desc, uint32_t T) {
  if (!desc_ok(desc)) return -1;
  Ctx c = make_ctx(desc, nullptr, T, nullptr, nullptr);
  if (T == 0 || fused_eligible(c) || !tc_possible(*desc, T) || !tc_supported(*desc)) return -1;
  return (desc->flags & MOE_FLAG_FORCE_TC) ? 0 : (int32_t)tc_min_rows_for(desc->routed_fmt);
}

const char *moe_layer_stage_name(const moe_desc *desc, uint32_t T, uint32_t i) {
  const char *path = moe_layer_path(desc, T);
  if (!path) return nullptr;
  if (path[0] == 'f') return i < kNumFusedStages ? kFusedStageNames[i] : nullptr;
  return i < kNumStages ? kStageNames[i] : nullptr;
}

moe_status moe_router_logits(const moe_desc *desc, const float *w_router, const float *x,
                             uint32_t T, float *logits, void *stream) {
  if (!desc_ok(desc)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!w_router || !x || !logits || !aligned(w_router, 16) || !aligned(x, 16) ||
      !aligned(logits, 4) || desc->d > 32768 || (uint64_t)T * desc->n_expert > 0x7fffffffull)
    return MOE_ERR_INVALID_ARG;
  return from_cuda(launch_router_logits(*desc, w_router, x, T, logits, (cudaStream_t)stream));
}

const char *moe_last_error(void) { return t_last_error; }

moe_status moe_check_device_error(void *ws, size_t ws_bytes, void *stream) {
  if (!ws) {
    // moe_layer_noalloc's static scratch on the current device (none before the
    // first such call there: then no kernel can have flagged anything)
    if (ws_bytes != 0) return MOE_ERR_INVALID_ARG;
    ws = noalloc_scratch_current();
    if (!ws) return MOE_OK;
    ws_bytes = MOE_NOALLOC_SCRATCH_BYTES;
  }
  if (ws_bytes < sizeof(uint32_t)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return from_cuda(e);
  if (word == 0) return MOE_OK;
  // the calls on `stream` have finished.  After a timeout the fused decode
  // kernel's counters may be left mid-count: zero the whole fixed head so the
  // workspace serves the next call; otherwise the error word alone
  const size_t clear =
      (word & kErrTimeout) && ws_bytes >= MOE_WS_FIXED_BYTES ? MOE_WS_FIXED_BYTES : sizeof word;
  e = cudaMemsetAsync(ws, 0, clear, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return from_cuda(e);
  return (word & kErrTimeout) ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE_CHECK;
}

const char *moe_status_string(moe_status st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device-side input check failed";
  }
  return "unknown status";
}

}  // extern "C"
