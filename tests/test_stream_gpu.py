"""Host-tier expert streaming on the GPU (pytest -m gpu).

Routed experts served from an HBM cache over pinned host memory (the pages'
expert streaming with an LFU cache and router-lookahead prefetch: NeutronStar
glm-local README, "SSD streaming optimizations") must give the same layer output,
bit for bit, as the same experts resident in HBM: the kernels read the same
bytes through the expert -> slot table (moe_weights.expert_slot); and a streamed
decode token and a streamed 16-row batch are also compared with the CPU oracle
directly."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from parity import compare_with_oracle, device_layer
from routed_expert_decode_gb300 import moe

pytestmark = pytest.mark.gpu

ROUTED = ("gate", "up", "down")


def _spec(**kw):
    base = dict(name="stream", E=16, k=4, d=512, f=256, f_shared=256, fmt=0, s=2.5,
                zipf_beta=0.4)
    base.update(kw)
    return synth.LayerSpec(**base)


def _mats(tensors, names):
    w = moe.MoeWeights()
    for n in names:
        setattr(w, n, moe.MoeMat(tensors[n + "_q"].data_ptr(), tensors[n + "_s"].data_ptr()))
    return w


def _slot_layer(layer, perm, n_slots, dev):
    """The layer's routed planes rearranged into n_slots slots: expert e in slot
    perm[e]; returns (weights with the slot table, tensors kept alive)."""
    t = layer.tensors
    keep = {}
    for n in ROUTED:
        for sfx in ("_q", "_s"):
            src = t[n + sfx]
            dst = torch.zeros((n_slots,) + tuple(src.shape[1:]), dtype=src.dtype, device=dev)
            dst[torch.as_tensor(perm, device=dev, dtype=torch.long)] = src
            keep[n + sfx] = dst
    w = moe.MoeWeights()
    for n in ROUTED:
        setattr(w, n, moe.MoeMat(keep[n + "_q"].data_ptr(), keep[n + "_s"].data_ptr()))
    for n in ("s_gate", "s_up", "s_down"):
        setattr(w, n, getattr(layer.weights, n))
    table = torch.as_tensor(np.asarray(perm, np.int32), device=dev)
    keep["table"] = table
    w.expert_slot = table.data_ptr()
    w.n_slots = n_slots
    return w, keep


@pytest.mark.parametrize("T,flags", [(1, 0), (2, 0), (6, 0), (40, 0), (40, "tc")],
                         ids=["fused_t1", "fused_t2", "gemv_t6", "mixed_t40", "tc_t40"])
def test_slot_table_gives_identical_output(gpu, T, flags):
    spec = _spec()
    layer = device_layer(spec, gpu)
    fl = moe.FLAG_FORCE_TC if flags == "tc" else 0
    desc = layer.desc(fl)
    n_slots = spec.E + 5
    perm = np.random.default_rng(T).permutation(n_slots)[:spec.E]
    w_slot, keep = _slot_layer(layer, perm, n_slots, gpu)
    logits, x = synth.token_inputs(spec, 9, T)
    args = [torch.from_numpy(a).to(gpu) for a in (x, logits, synth.bias(spec))]
    ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=gpu)
    y_ref = torch.empty((T, spec.d), dtype=torch.float32, device=gpu)
    y_slot = torch.empty_like(y_ref)
    moe.layer(desc, layer.weights, *args[:2], args[2], y_ref, ws)
    moe.layer(desc, w_slot, *args[:2], args[2], y_slot, ws)
    torch.cuda.synchronize()
    assert moe.check_device_error(ws) == 0
    assert torch.equal(y_ref, y_slot)


@pytest.mark.parametrize("T", [1, 2, 6])
def test_selected_expert_outside_the_slots_is_a_device_error(gpu, T):
    """A selected expert whose slot is >= n_slots fails the device check; no
    weight row outside the slots is read (the kernels plan no routed work).
    On the fused decode kernel (T <= 2) every CTA routes and may flag the bad
    slot before any other has started, so the call is repeated 50 times: the
    flag must never be lost."""
    spec = _spec()
    layer = device_layer(spec, gpu)
    desc = layer.desc()
    n_slots = spec.E
    perm = np.arange(spec.E)
    w_slot, keep = _slot_layer(layer, perm, n_slots, gpu)
    logits, x = synth.token_inputs(spec, 3, T)
    picks, _ = __import__("oracle").route(logits, synth.bias(spec), spec.k, spec.s)
    keep["table"][int(picks[0, 0])] = n_slots  # out of range for a selected expert
    ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=gpu)
    y = torch.empty((T, spec.d), dtype=torch.float32, device=gpu)
    assert moe.layer_path(desc, T) == ("fused_decode" if T <= 2 else "multi_kernel")
    for _ in range(50 if T <= 2 else 1):
        moe.layer(desc, w_slot, torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu),
                  torch.from_numpy(synth.bias(spec)).to(gpu), y, ws)
        torch.cuda.synchronize()
        assert moe.STATUS_NAMES[moe.check_device_error(ws)] == "MOE_ERR_DEVICE_CHECK"
    # the workspace stays usable
    keep["table"][int(picks[0, 0])] = int(perm[int(picks[0, 0])])
    moe.layer(desc, w_slot, torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu),
              torch.from_numpy(synth.bias(spec)).to(gpu), y, ws)
    torch.cuda.synchronize()
    assert moe.check_device_error(ws) == 0


class StreamedStack:
    """L layers whose routed experts live in pinned host memory, served by one
    HBM cache of n_slots slots; the shared experts stay resident."""

    def __init__(self, specs, n_slots, dev):
        self.specs = specs
        self.dev = dev
        self.layers = []
        self.host = []
        self.keep = []
        for s in specs:
            t = synth.fill_layer_device(s, dev)
            lay = moe.Layer(s.E, s.k, s.d, s.f, s.f_shared, s.fmt, s.s, t, dev)
            host_t = {n + sfx: t[n + sfx].cpu().pin_memory() for n in ROUTED for sfx in ("_q", "_s")}
            self.host.append(_mats(host_t, ROUTED))
            self.keep.append(host_t)
            self.layers.append(lay)
        s0 = specs[0]
        self.arena_t = {}
        for n in ROUTED:
            for sfx in ("_q", "_s"):
                src = self.layers[0].tensors[n + sfx]
                self.arena_t[n + sfx] = torch.zeros((n_slots,) + tuple(src.shape[1:]),
                                                    dtype=src.dtype, device=dev)
        self.arena = _mats(self.arena_t, ROUTED)
        self.table = torch.full((len(specs), s0.E), -1, dtype=torch.int32, device=dev)
        self.desc = self.layers[0].desc()
        self.cache = moe.ExpertCache(self.desc, self.host, self.arena, n_slots,
                                     self.table.data_ptr())

    def shared(self, l):
        w = moe.MoeWeights()
        for n in ("s_gate", "s_up", "s_down"):
            setattr(w, n, getattr(self.layers[l].weights, n))
        return w


@pytest.mark.parametrize("lookahead", [False, True], ids=["demand", "lookahead"])
def test_streamed_layers_match_resident(gpu, lookahead):
    L, T = 3, 2
    specs = [dataclasses.replace(_spec(), name=f"stream{l}", layer_seed=100 + l) for l in range(L)]
    st = StreamedStack(specs, n_slots=12, dev=gpu)
    side = torch.cuda.Stream(gpu)
    ws = torch.zeros(moe.workspace_size(st.desc, T), dtype=torch.uint8, device=gpu)
    ws_ref = torch.zeros_like(ws)
    biases = [torch.from_numpy(synth.bias(s)).to(gpu) for s in specs]
    for step in range(6):
        inputs = [synth.token_inputs(s, 50 + step, T) for s in specs]
        lg = [torch.from_numpy(a[0]).to(gpu) for a in inputs]
        xs = [torch.from_numpy(a[1]).to(gpu) for a in inputs]
        for l in range(L):
            y = torch.empty((T, specs[l].d), dtype=torch.float32, device=gpu)
            nxt = lookahead and l + 1 < L
            moe.stream_layer(st.cache, l, st.desc, st.shared(l), xs[l], lg[l], biases[l], y, ws,
                             next_logits=lg[l + 1] if nxt else None,
                             next_bias=biases[l + 1] if nxt else None, prefetch_stream=side)
            y_ref = torch.empty_like(y)
            moe.layer(st.layers[l].desc(), st.layers[l].weights, xs[l], lg[l], biases[l], y_ref,
                      ws_ref)
            torch.cuda.synchronize()
            assert moe.check_device_error(ws) == 0
            assert torch.equal(y, y_ref), f"step {step} layer {l}"
            # the device table agrees with the cache for this layer's picks
            tab = st.table[l].cpu().numpy()
            picks = st.layers[l].views(ws_ref, T)["idx"].cpu().numpy().reshape(-1)
            for e in picks:
                assert tab[e] == st.cache.slot(l, int(e)) >= 0
    stats = st.cache.stats()
    assert stats["lookups"] == stats["hits"] + stats["misses"]
    assert stats["misses"] > 0 and stats["evictions"] > 0
    if lookahead:
        assert stats["prefetch_loads"] > 0 and stats["prefetch_hits"] > 0
    st.cache.close()


def test_streamed_full_size_decode_matches_resident(gpu):
    """The full-size layer (E=256, top-8, d=6144, f=2048, shared 2048, Q8_0)
    streamed from pinned host memory through an 18-slot cache, two layers
    sharing the routed bytes as in the bench's stack, one token per call, with
    the lookahead prefetch: bit-identical to the same layer resident in HBM."""
    spec = synth.GLM_LAYER
    layer = device_layer(spec, gpu)
    host_t = {n + sfx: layer.tensors[n + sfx].cpu().pin_memory()
              for n in ROUTED for sfx in ("_q", "_s")}
    host_w = _mats(host_t, ROUTED)
    n_slots = 18
    arena_t = {k: torch.zeros((n_slots,) + tuple(v.shape[1:]), dtype=v.dtype, device=gpu)
               for k, v in host_t.items()}
    arena = _mats(arena_t, ROUTED)
    table = torch.full((2, spec.E), -1, dtype=torch.int32, device=gpu)
    desc = layer.desc()
    cache = moe.ExpertCache(desc, [host_w, host_w], arena, n_slots, table.data_ptr())
    shared = moe.MoeWeights()
    for n in ("s_gate", "s_up", "s_down"):
        setattr(shared, n, getattr(layer.weights, n))
    bias = torch.from_numpy(synth.bias(spec)).to(gpu)
    ws = torch.zeros(moe.workspace_size(desc, 1), dtype=torch.uint8, device=gpu)
    ws_ref = torch.zeros_like(ws)
    side = torch.cuda.Stream(gpu)
    for tok in range(3):
        ins = [synth.token_inputs(spec, 300 + tok + 100 * l, 1) for l in range(2)]
        lg = [torch.from_numpy(i[0]).to(gpu) for i in ins]
        xs = [torch.from_numpy(i[1]).to(gpu) for i in ins]
        for l in range(2):
            y = torch.empty((1, spec.d), dtype=torch.float32, device=gpu)
            y_ref = torch.empty_like(y)
            moe.stream_layer(cache, l, desc, shared, xs[l], lg[l], bias, y, ws,
                             next_logits=lg[1] if l == 0 else None,
                             next_bias=bias if l == 0 else None, prefetch_stream=side)
            moe.layer(desc, layer.weights, xs[l], lg[l], bias, y_ref, ws_ref)
            torch.cuda.synchronize()
            assert moe.check_device_error(ws) == 0
            assert torch.equal(y, y_ref), f"token {tok} layer {l}"
    st = cache.stats()
    assert st["misses"] > 0 and st["lookups"] == st["hits"] + st["misses"]
    cache.close()


@pytest.mark.parametrize("T", [1, 16])
def test_streamed_layer_matches_oracle(gpu, T):
    """The decode-shaped layer (d=6144, f=2048, shared 2048, Q8_0; 32 experts)
    with its routed experts in pinned host memory, served through a cold HBM
    cache: idx, off, perm, xq exact and y within tolerance against the CPU
    oracle (T=1 on the fused kernel, T=16 on the multi-kernel path)."""
    spec = synth.GLM_LAYER_E32
    layer = device_layer(spec, gpu)
    host_t = {n + sfx: layer.tensors[n + sfx].cpu().pin_memory()
              for n in ROUTED for sfx in ("_q", "_s")}
    n_slots = spec.E
    arena_t = {k: torch.zeros((n_slots,) + tuple(v.shape[1:]), dtype=v.dtype, device=gpu)
               for k, v in host_t.items()}
    table = torch.full((1, spec.E), -1, dtype=torch.int32, device=gpu)
    desc = layer.desc()
    cache = moe.ExpertCache(desc, [_mats(host_t, ROUTED)], _mats(arena_t, ROUTED), n_slots,
                            table.data_ptr())
    shared = moe.MoeWeights()
    for n in ("s_gate", "s_up", "s_down"):
        setattr(shared, n, getattr(layer.weights, n))
    bias = synth.bias(spec)
    ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=gpu)
    for seed in (61, 62):
        logits, x = synth.token_inputs(spec, seed, T)
        y = torch.empty((T, spec.d), dtype=torch.float32, device=gpu)
        moe.stream_layer(cache, 0, desc, shared, torch.from_numpy(x).to(gpu),
                         torch.from_numpy(logits).to(gpu), torch.from_numpy(bias).to(gpu), y, ws)
        torch.cuda.synchronize()
        assert moe.check_device_error(ws) == 0
        v = layer.views(ws, T)
        g = {k: (t.cpu().numpy() if isinstance(t, torch.Tensor) else t) for k, t in v.items()}
        g["y"] = y.cpu().numpy()
        rep = compare_with_oracle(spec, T, x, logits, bias, g,
                                  sample=None if T == 1 else [0, 7, 15])
        print("streamed", T, seed, rep)
    st = cache.stats()
    assert st["misses"] > 0
    cache.close()
