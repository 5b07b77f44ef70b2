// expert_cache.cu -- an HBM expert cache over a host tier (moe_cache_*, moe.h).
//
// The pages stream routed experts from a slower tier into a GPU-side cache:
// popularity is concentrated enough that an LFU cache of the hottest experts
// removes a large share of the slow-tier traffic, a batch loads the union of its
// experts once, and the next layer's router is run early so that its experts can
// be fetched while the current layer computes (NeutronStar glm-local README,
// "SSD streaming optimizations"; NeutronStar README, the host-cache and
// cross-layer prefetch paragraphs).  On GB300 the slow tier is host memory
// (Grace LPDDR, pinned) across NVLink-C2C and the cache is an arena of expert
// slots in HBM shared by every layer; the copies are plain cudaMemcpyAsync calls
// on the copy engines, one per weight plane of a loaded expert.
//
// Host-only code: the policy is deterministic and needs no device (the
// MOE_CACHE_POLICY_ONLY mode and moe_cache_plan run it without CUDA), the copies
// and events are ordered as moe.h states.
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include "moe_internal.cuh"

struct moe_cache {
  moe_desc desc;
  uint32_t L = 0, E = 0, S = 0;
  uint32_t flags = 0;
  std::vector<moe_weights> host;   // per layer: routed planes in host memory
  moe_weights arena;               // routed planes with S slots in HBM
  int32_t *d_table = nullptr;      // device [L][E]
  std::vector<int32_t> slot_of;    // [L*E]: slot or -1
  std::vector<int64_t> owner;      // [S]: L*E id or -1
  std::vector<uint64_t> count;     // [L*E]: lookups (LFU frequency), kept across evictions
  std::vector<uint64_t> last;      // [L*E]: stamp of the latest lookup
  std::vector<uint8_t> prefetched; // [L*E]: loaded by a prefetch, not yet looked up
  std::vector<uint8_t> pending;    // [S]: a prefetch copy into the slot may be in flight
  std::vector<cudaEvent_t> ready;  // [S]: recorded after a prefetch's copies into the slot
  std::vector<uint8_t> busy;       // [L*E]: named by the latest ensure
  std::vector<int64_t> busy_list;
  cudaEvent_t after_latest = nullptr;  // compute stream, after the latest ensure's copies
  bool have_latest = false;
  uint64_t stamp = 0;
  moe_cache_stats st;
  std::vector<int32_t> table_stage;  // [E] host staging of a layer's slot table
  int32_t *pinned = nullptr;         // pinned host buffer for moe_stream_layer's read-back
  size_t pinned_n = 0;
};

namespace moe {
namespace {

struct Load {
  int32_t expert;
  int32_t slot;
  int64_t evicted;
};

size_t gu_q_bytes(const moe_desc &D) { return (size_t)D.f * row_bytes(D.routed_fmt, D.d); }
size_t gu_s_bytes(const moe_desc &D) { return (size_t)D.f * (D.d / 32) * 2; }
size_t dn_q_bytes(const moe_desc &D) { return (size_t)D.d * row_bytes(D.routed_fmt, D.f); }
size_t dn_s_bytes(const moe_desc &D) { return (size_t)D.d * (D.f / 32) * 2; }
size_t expert_bytes(const moe_desc &D) {
  return 2 * (gu_q_bytes(D) + gu_s_bytes(D)) + dn_q_bytes(D) + dn_s_bytes(D);
}

// the distinct experts of experts[0..n) in ascending order; false on one out of range
bool distinct(const moe_cache &c, const int32_t *experts, uint32_t n, std::vector<int32_t> *u) {
  u->clear();
  for (uint32_t i = 0; i < n; ++i) {
    if (experts[i] < 0 || (uint32_t)experts[i] >= c.E) return false;
    u->push_back(experts[i]);
  }
  std::sort(u->begin(), u->end());
  u->erase(std::unique(u->begin(), u->end()), u->end());
  return true;
}

// LFU victim: fewest lookups, then least recent use, then lower id; never a
// protected expert.  -1 when every slot is protected.
int32_t pick_victim(const moe_cache &c, const std::vector<uint8_t> &protect) {
  int32_t best = -1;
  for (uint32_t s = 0; s < c.S; ++s) {
    const int64_t g = c.owner[s];
    if (g < 0 || protect[g]) continue;
    if (best < 0) {
      best = (int32_t)s;
      continue;
    }
    const int64_t b = c.owner[best];
    if (c.count[g] < c.count[b] ||
        (c.count[g] == c.count[b] &&
         (c.last[g] < c.last[b] || (c.last[g] == c.last[b] && g < b))))
      best = (int32_t)s;
  }
  return best;
}

int32_t free_slot(const moe_cache &c) {
  for (uint32_t s = 0; s < c.S; ++s)
    if (c.owner[s] < 0) return (int32_t)s;
  return -1;
}

// The policy step shared by ensure, prefetch and plan: decides the loads and
// updates the state.  A demand call that cannot place its whole union changes
// nothing and fails; a prefetch stops at the first expert it cannot place.
moe_status decide(moe_cache &c, uint32_t layer, const int32_t *experts, uint32_t n,
                  bool prefetch, std::vector<Load> *loads, std::vector<int32_t> *hits_pending) {
  loads->clear();
  if (hits_pending) hits_pending->clear();
  if (layer >= c.L) return MOE_ERR_INVALID_ARG;
  std::vector<int32_t> u;
  if (!distinct(c, experts, n, &u)) return MOE_ERR_INVALID_ARG;
  const int64_t base = (int64_t)layer * c.E;
  std::vector<uint8_t> protect(c.slot_of.size(), 0);
  for (int32_t e : u) protect[base + e] = 1;
  if (prefetch)
    for (int64_t g : c.busy_list) protect[g] = 1;
  if (!prefetch) {
    // the whole union must fit: count what is missing against what may go
    uint32_t missing = 0, movable = 0;
    for (int32_t e : u) missing += c.slot_of[base + e] < 0 ? 1u : 0u;
    for (uint32_t s = 0; s < c.S; ++s)
      if (c.owner[s] < 0 || !protect[c.owner[s]]) ++movable;
    if (missing > movable) return MOE_ERR_WORKSPACE;
  }
  for (int32_t e : u) {
    const int64_t g = base + e;
    if (!prefetch) {
      c.count[g] += 1;
      c.last[g] = ++c.stamp;
      c.st.lookups += 1;
    }
    if (c.slot_of[g] >= 0) {
      if (!prefetch) {
        c.st.hits += 1;
        if (c.prefetched[g]) {
          c.st.prefetch_hits += 1;
          c.prefetched[g] = 0;
        }
        if (hits_pending && c.pending[c.slot_of[g]]) hits_pending->push_back(c.slot_of[g]);
      }
      continue;
    }
    int32_t s = free_slot(c);
    int64_t victim = -1;
    if (s < 0) {
      s = pick_victim(c, protect);
      if (s < 0) break;  // prefetch only: nothing more may be evicted
      victim = c.owner[s];
      c.slot_of[victim] = -1;
      c.prefetched[victim] = 0;
      c.st.evictions += 1;
    }
    c.owner[s] = g;
    c.slot_of[g] = s;
    c.prefetched[g] = prefetch ? 1 : 0;
    if (prefetch) c.st.prefetch_loads += 1;
    else c.st.misses += 1;
    c.st.bytes_h2d += expert_bytes(c.desc);
    loads->push_back(Load{e, s, victim});
  }
  if (!prefetch) {
    for (int64_t g : c.busy_list) c.busy[g] = 0;
    c.busy_list.clear();
    for (int32_t e : u) {
      c.busy[base + e] = 1;
      c.busy_list.push_back(base + e);
    }
  }
  return MOE_OK;
}

// the six plane copies of one expert into its slot
cudaError_t copy_expert(const moe_cache &c, uint32_t layer, int32_t e, int32_t s,
                        cudaStream_t st) {
  const moe_desc &D = c.desc;
  const moe_weights &h = c.host[layer];
  const size_t gq = gu_q_bytes(D), gs = gu_s_bytes(D), dq = dn_q_bytes(D), ds = dn_s_bytes(D);
  struct Plane {
    const void *src;
    void *dst;
    size_t bytes;
  } planes[6] = {
      {h.gate.q, (void *)c.arena.gate.q, gq},     {h.gate.scale, (void *)c.arena.gate.scale, gs},
      {h.up.q, (void *)c.arena.up.q, gq},         {h.up.scale, (void *)c.arena.up.scale, gs},
      {h.down.q, (void *)c.arena.down.q, dq},     {h.down.scale, (void *)c.arena.down.scale, ds},
  };
  for (const Plane &p : planes) {
    const uint8_t *src = (const uint8_t *)p.src + (size_t)e * p.bytes;
    uint8_t *dst = (uint8_t *)p.dst + (size_t)s * p.bytes;
    cudaError_t err = cudaMemcpyAsync(dst, src, p.bytes, cudaMemcpyHostToDevice, st);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t upload_table(moe_cache &c, uint32_t layer, cudaStream_t st) {
  const size_t base = (size_t)layer * c.E;
  for (uint32_t e = 0; e < c.E; ++e) c.table_stage[e] = c.slot_of[base + e];
  // pageable source: staged by the driver before the call returns
  return cudaMemcpyAsync(c.d_table + base, c.table_stage.data(), (size_t)c.E * 4,
                         cudaMemcpyHostToDevice, st);
}

bool mats_ok(const moe_weights &w) {
  return w.gate.q && w.gate.scale && w.up.q && w.up.scale && w.down.q && w.down.scale;
}

}  // namespace

// internal accessors for moe_stream_layer (moe_api.cu)
bool cache_layer_routed(const moe_cache *c, uint32_t layer, moe_weights *w) {
  if (!c || layer >= c->L) return false;
  w->gate = c->arena.gate;
  w->up = c->arena.up;
  w->down = c->arena.down;
  w->expert_slot = c->d_table + (size_t)layer * c->E;
  w->n_slots = c->S;
  return true;
}

const moe_desc *cache_desc(const moe_cache *c) { return c ? &c->desc : nullptr; }

int32_t *cache_pinned(moe_cache *c, size_t n) {
  if (c->pinned_n < n) {
    if (c->pinned) cudaFreeHost(c->pinned);
    c->pinned = nullptr;
    c->pinned_n = 0;
    void *p = nullptr;
    if (cudaHostAlloc(&p, n * 4, cudaHostAllocDefault) != cudaSuccess) return nullptr;
    c->pinned = (int32_t *)p;
    c->pinned_n = n;
  }
  return c->pinned;
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_cache_create(const moe_desc *desc, uint32_t n_layers,
                            const moe_weights *host_layers, const moe_weights *arena,
                            uint32_t n_slots, int32_t *slot_table, uint32_t flags,
                            moe_cache **out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!desc || !host_layers || !arena || !slot_table || n_layers == 0 || n_slots == 0)
    return MOE_ERR_INVALID_ARG;
  if (moe_workspace_size(desc, 1) == 0) return MOE_ERR_INVALID_ARG;  // desc check
  if (flags & ~MOE_CACHE_POLICY_ONLY) return MOE_ERR_INVALID_ARG;
  if ((uint64_t)n_layers * desc->n_expert > (1u << 24)) return MOE_ERR_INVALID_ARG;
  if (!mats_ok(*arena)) return MOE_ERR_INVALID_ARG;
  for (uint32_t l = 0; l < n_layers; ++l)
    if (!mats_ok(host_layers[l])) return MOE_ERR_INVALID_ARG;
  moe_cache *c = new (std::nothrow) moe_cache();
  if (!c) return MOE_ERR_WORKSPACE;
  c->desc = *desc;
  c->L = n_layers;
  c->E = desc->n_expert;
  c->S = n_slots;
  c->flags = flags;
  c->host.assign(host_layers, host_layers + n_layers);
  c->arena = *arena;
  c->d_table = slot_table;
  const size_t G = (size_t)n_layers * c->E;
  c->slot_of.assign(G, -1);
  c->owner.assign(n_slots, -1);
  c->count.assign(G, 0);
  c->last.assign(G, 0);
  c->prefetched.assign(G, 0);
  c->busy.assign(G, 0);
  c->pending.assign(n_slots, 0);
  c->table_stage.assign(c->E, -1);
  memset(&c->st, 0, sizeof c->st);
  if (!(flags & MOE_CACHE_POLICY_ONLY)) {
    c->ready.assign(n_slots, nullptr);
    bool ok = cudaEventCreateWithFlags(&c->after_latest, cudaEventDisableTiming) == cudaSuccess;
    for (uint32_t s = 0; s < n_slots && ok; ++s)
      ok = cudaEventCreateWithFlags(&c->ready[s], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      moe_cache_destroy(c);
      set_last_error("moe_cache_create: cudaEventCreate failed");
      return MOE_ERR_CUDA;
    }
  }
  *out = c;
  return MOE_OK;
}

void moe_cache_destroy(moe_cache *c) {
  if (!c) return;
  for (cudaEvent_t ev : c->ready)
    if (ev) cudaEventDestroy(ev);
  if (c->after_latest) cudaEventDestroy(c->after_latest);
  if (c->pinned) cudaFreeHost(c->pinned);
  delete c;
}

moe_status moe_cache_plan(moe_cache *c, uint32_t layer, const int32_t *experts, uint32_t n,
                          int prefetch, int32_t *loaded, int32_t *slots, int64_t *evicted,
                          uint32_t *n_loaded) {
  if (!c || (n && !experts) || !n_loaded || (n && (!loaded || !slots || !evicted)))
    return MOE_ERR_INVALID_ARG;
  std::vector<Load> loads;
  const moe_status st = decide(*c, layer, experts, n, prefetch != 0, &loads, nullptr);
  if (st != MOE_OK) return st;
  for (size_t i = 0; i < loads.size(); ++i) {
    loaded[i] = loads[i].expert;
    slots[i] = loads[i].slot;
    evicted[i] = loads[i].evicted;
  }
  *n_loaded = (uint32_t)loads.size();
  return MOE_OK;
}

moe_status moe_cache_ensure(moe_cache *c, uint32_t layer, const int32_t *experts, uint32_t n,
                            void *stream) {
  if (!c || (n && !experts)) return MOE_ERR_INVALID_ARG;
  if (c->flags & MOE_CACHE_POLICY_ONLY) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  std::vector<Load> loads;
  std::vector<int32_t> wait_slots;
  moe_status s = decide(*c, layer, experts, n, false, &loads, &wait_slots);
  if (s != MOE_OK) return s;
  cudaError_t e = cudaSuccess;
  // hits still arriving by a prefetch, and slots a prefetch may still be writing
  for (int32_t slot : wait_slots)
    if (e == cudaSuccess) {
      e = cudaStreamWaitEvent(st, c->ready[slot], 0);
      c->pending[slot] = 0;
    }
  for (const Load &ld : loads) {
    if (e == cudaSuccess && c->pending[ld.slot]) {
      e = cudaStreamWaitEvent(st, c->ready[ld.slot], 0);
      c->pending[ld.slot] = 0;
    }
    if (e == cudaSuccess) e = copy_expert(*c, layer, ld.expert, ld.slot, st);
  }
  if (e == cudaSuccess) e = upload_table(*c, layer, st);
  // later prefetches start after these copies: the layer's own misses get the
  // link first, and every compute use of a slot enqueued before is behind them
  if (e == cudaSuccess) e = cudaEventRecord(c->after_latest, st);
  c->have_latest = e == cudaSuccess;
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorName(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status moe_cache_prefetch(moe_cache *c, uint32_t layer, const int32_t *experts, uint32_t n,
                              void *stream) {
  if (!c || (n && !experts)) return MOE_ERR_INVALID_ARG;
  if (c->flags & MOE_CACHE_POLICY_ONLY) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  std::vector<Load> loads;
  moe_status s = decide(*c, layer, experts, n, true, &loads, nullptr);
  if (s != MOE_OK) return s;
  cudaError_t e = cudaSuccess;
  // start after the latest ensure's copies: its misses go first on the link, and
  // an evicted expert's slot is no longer read by compute work enqueued before it
  if (!loads.empty() && c->have_latest) e = cudaStreamWaitEvent(st, c->after_latest, 0);
  for (const Load &ld : loads) {
    if (e == cudaSuccess && c->pending[ld.slot]) e = cudaStreamWaitEvent(st, c->ready[ld.slot], 0);
    if (e == cudaSuccess) e = copy_expert(*c, layer, ld.expert, ld.slot, st);
    if (e == cudaSuccess) e = cudaEventRecord(c->ready[ld.slot], st);
    if (e == cudaSuccess) c->pending[ld.slot] = 1;
  }
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorName(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

uint32_t moe_cache_layers(const moe_cache *c) { return c ? c->L : 0u; }

int32_t moe_cache_slot(const moe_cache *c, uint32_t layer, int32_t expert) {
  if (!c || layer >= c->L || expert < 0 || (uint32_t)expert >= c->E) return -1;
  return c->slot_of[(size_t)layer * c->E + expert];
}

moe_status moe_cache_get_stats(const moe_cache *c, moe_cache_stats *out) {
  if (!c || !out) return MOE_ERR_INVALID_ARG;
  *out = c->st;
  return MOE_OK;
}

}  // extern "C"
