"""Python binding of ``libmoe.so`` (C ABI in ``include/moe.h``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.  There is no
CPU fallback: if the library is missing or the tensors are not on a CUDA
device, the call raises.

Entry points mirror the C names: ``workspace_size``, ``workspace_layout``,
``route``, ``ffn``, ``layer``, ``check_device_error``, ``status_string``.
``Layer`` bundles one layer's weights, descriptor and workspace.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT",
                6: "MOE_ERR_DEVICE_CHECK"}
FMT_Q8_0 = 0
FMT_Q2S = 1
FMT_E2M1 = 2
FLAG_DEBUG_TAPS = 0x1
FLAG_FORCE_GEMV = 0x2
FLAG_FORCE_TC = 0x4
FLAG_TEST_STALL = 0x8
FLAG_TRACE = 0x10
TRACE_FIELDS = ("start_ns", "xq_done_ns", "first_stage_ns", "wait_full_cyc", "wait_ready_cyc",
                "stages_b", "stages_c", "cons_end_ns", "wait_empty_cyc", "wait_route_cyc",
                "items", "compute_b_cyc", "compute_c_cyc", "combine_cyc", "route_done_ns",
                "prod_end_ns", "route_loaded_ns", "route_topk_ns", "route_perm_ns", "exit_ns",
                "w5_wait_full_cyc", "w5_compute_b_cyc", "w5_compute_c_cyc", "item_end_cyc",
                "select_topk_ns", "select_weights_ns", "select_perm_ns", "router_written_ns",
                "lat_issue_got_cyc", "lat_got_rel_cyc", "lat_rel_empty_cyc", "lat_samples")

_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_u32 = ctypes.c_uint32


class MoeMat(ctypes.Structure):
    _fields_ = [("q", _vp), ("scale", _vp)]


class MoeDesc(ctypes.Structure):
    _fields_ = [("n_expert", _u32), ("top_k", _u32), ("d", _u32), ("f", _u32),
                ("f_shared", _u32), ("routed_fmt", ctypes.c_int32), ("s", ctypes.c_float),
                ("flags", _u32), ("score", _u32)]


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, MoeMat) for n in ("gate", "up", "down", "s_gate", "s_up", "s_down")] + \
        [("expert_slot", _vp), ("n_slots", _u32)]


LAYOUT_FIELDS = ("idx", "w", "off", "perm", "pos", "xq", "xs", "hq", "hs", "h", "o", "plan",
                 "sync", "tap_gu", "tap_dn", "trace", "xperm", "xsperm", "hperm", "xt", "ht", "rseg",
                 "lidx", "lw", "err",
                 "total")


class MoeWsLayout(ctypes.Structure):
    _fields_ = [(n, _sz) for n in LAYOUT_FIELDS] + [("n_tap", _u32)]


class MoeCacheStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("lookups", "hits", "misses", "prefetch_loads",
                                               "prefetch_hits", "evictions", "bytes_h2d")]


CACHE_POLICY_ONLY = 1


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        detail = status_string(status) if _lib else ""
        if status == 4 and _lib:
            detail += ": " + _lib.moe_last_error().decode()
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({detail})")
        self.status = status


_lib = None


def lib():
    """Load libmoe.so; raise (never fall back) if it is absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.moe_workspace_size.restype = _sz
        L.moe_workspace_size.argtypes = [ctypes.POINTER(MoeDesc), _u32]
        L.moe_workspace_layout.restype = ctypes.c_int
        L.moe_workspace_layout.argtypes = [ctypes.POINTER(MoeDesc), _u32,
                                           ctypes.POINTER(MoeWsLayout)]
        L.moe_route.restype = ctypes.c_int
        L.moe_route.argtypes = [ctypes.POINTER(MoeDesc), _vp, _vp, _u32, _vp, _vp, _vp, _vp, _vp,
                                _vp, _sz, _vp]
        L.moe_ffn.restype = ctypes.c_int
        L.moe_ffn.argtypes = [ctypes.POINTER(MoeDesc), ctypes.POINTER(MoeWeights), _vp, _u32,
                              _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
        L.moe_layer.restype = ctypes.c_int
        L.moe_layer.argtypes = [ctypes.POINTER(MoeDesc), ctypes.POINTER(MoeWeights), _vp, _vp,
                                _vp, _u32, _vp, _vp, _sz, _vp]
        L.moe_layer_timed.restype = ctypes.c_int
        L.moe_layer_timed.argtypes = [ctypes.POINTER(MoeDesc), ctypes.POINTER(MoeWeights), _vp,
                                      _vp, _vp, _u32, _vp, _vp, _sz, _vp,
                                      ctypes.POINTER(_vp), _u32]
        L.moe_layer_path.restype = ctypes.c_char_p
        L.moe_layer_path.argtypes = [ctypes.POINTER(MoeDesc), _u32]
        L.moe_router_logits.argtypes = [ctypes.POINTER(MoeDesc), _vp, _vp, _u32, _vp, _vp]
        L.moe_router_logits.restype = ctypes.c_int
        L.moe_layer_from_x.argtypes = [ctypes.POINTER(MoeDesc), ctypes.POINTER(MoeWeights), _vp,
                                       _vp, _vp, _u32, _vp, _vp, _vp, _sz, _vp]
        L.moe_layer_from_x.restype = ctypes.c_int
        L.moe_layer_stage_name.restype = ctypes.c_char_p
        L.moe_tc_min_rows.argtypes = [ctypes.POINTER(MoeDesc), _u32]
        L.moe_tc_min_rows.restype = ctypes.c_int32
        L.moe_layer_stage_name.argtypes = [ctypes.POINTER(MoeDesc), _u32, _u32]
        L.moe_layer_experts.restype = ctypes.c_int
        L.moe_layer_experts.argtypes = [ctypes.POINTER(MoeDesc), ctypes.POINTER(MoeWeights), _vp,
                                        _vp, _vp, _u32, _u32, _u32, ctypes.c_int32, _vp, _vp, _sz,
                                        _vp]
        L.moe_ffn_experts.restype = ctypes.c_int
        L.moe_ffn_experts.argtypes = [ctypes.POINTER(MoeDesc), ctypes.POINTER(MoeWeights), _vp,
                                      _u32, _vp, _vp, _vp, _vp, _vp, _u32, _u32, ctypes.c_int32,
                                      _vp, _vp, _sz, _vp]
        L.moe_layer_noalloc.restype = ctypes.c_int
        L.moe_layer_noalloc.argtypes = [ctypes.POINTER(MoeDesc), ctypes.POINTER(MoeWeights), _vp,
                                        _vp, _vp, _u32, _vp, _vp]
        _pc = ctypes.POINTER(ctypes.c_void_p)
        L.moe_cache_create.restype = ctypes.c_int
        L.moe_cache_create.argtypes = [ctypes.POINTER(MoeDesc), _u32, ctypes.POINTER(MoeWeights),
                                       ctypes.POINTER(MoeWeights), _u32, _vp, _u32, _pc]
        L.moe_cache_destroy.restype = None
        L.moe_cache_destroy.argtypes = [_vp]
        L.moe_cache_ensure.restype = ctypes.c_int
        L.moe_cache_ensure.argtypes = [_vp, _u32, _vp, _u32, _vp]
        L.moe_cache_prefetch.restype = ctypes.c_int
        L.moe_cache_prefetch.argtypes = [_vp, _u32, _vp, _u32, _vp]
        L.moe_cache_plan.restype = ctypes.c_int
        L.moe_cache_plan.argtypes = [_vp, _u32, _vp, _u32, ctypes.c_int, _vp, _vp, _vp,
                                     ctypes.POINTER(_u32)]
        L.moe_cache_slot.restype = ctypes.c_int32
        L.moe_cache_slot.argtypes = [_vp, _u32, ctypes.c_int32]
        L.moe_cache_layers.restype = _u32
        L.moe_cache_layers.argtypes = [_vp]
        L.moe_cache_get_stats.restype = ctypes.c_int
        L.moe_cache_get_stats.argtypes = [_vp, ctypes.POINTER(MoeCacheStats)]
        L.moe_stream_layer.restype = ctypes.c_int
        L.moe_stream_layer.argtypes = [_vp, _u32, ctypes.POINTER(MoeDesc),
                                       ctypes.POINTER(MoeWeights), _vp, _vp, _vp, _u32, _vp, _vp,
                                       _vp, _vp, _sz, _vp, _vp]
        L.moe_check_device_error.restype = ctypes.c_int
        L.moe_check_device_error.argtypes = [_vp, _sz, _vp]
        L.moe_last_error.restype = ctypes.c_char_p
        L.moe_last_error.argtypes = []
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev_ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status)


SCORE_SIGMOID = 0
SCORE_SQRT_SOFTPLUS = 1


def make_desc(n_expert, top_k, d, f, f_shared, routed_fmt, s, flags=0,
              score=SCORE_SIGMOID) -> MoeDesc:
    return MoeDesc(n_expert, top_k, d, f, f_shared, routed_fmt, float(s), flags, score)


def router_logits(desc: MoeDesc, w_router: torch.Tensor, x: torch.Tensor,
                  logits: torch.Tensor, stream=None) -> None:
    """logits[T][E] = x[T][d] . w_router[E][d]^T in the library's fixed fp32 order."""
    T = x.shape[0]
    st = lib().moe_router_logits(ctypes.byref(desc), _dev_ptr(w_router, torch.float32, "w_router"),
                                 _dev_ptr(x, torch.float32, "x"), T,
                                 _dev_ptr(logits, torch.float32, "logits"), _stream(stream))
    _check("moe_router_logits", st)


def workspace_size(desc: MoeDesc, T: int) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(desc), T))


def workspace_layout(desc: MoeDesc, T: int) -> MoeWsLayout:
    out = MoeWsLayout()
    _check("moe_workspace_layout", lib().moe_workspace_layout(ctypes.byref(desc), T,
                                                              ctypes.byref(out)))
    return out


def route(desc: MoeDesc, logits, bias, idx, w, off, perm, pos, stream=None):
    T = logits.shape[0] if logits is not None else 0
    st = lib().moe_route(ctypes.byref(desc), _dev_ptr(logits, torch.float32, "logits"),
                         _dev_ptr(bias, torch.float32, "bias"), T,
                         _dev_ptr(idx, torch.int32, "idx"), _dev_ptr(w, torch.float32, "w"),
                         _dev_ptr(off, torch.int32, "off"), _dev_ptr(perm, torch.int32, "perm"),
                         _dev_ptr(pos, torch.int32, "pos"), None, 0, _stream(stream))
    _check("moe_route", st)


def ffn(desc: MoeDesc, weights: MoeWeights, x, idx, w, off, perm, pos, y, ws, stream=None):
    st = lib().moe_ffn(ctypes.byref(desc), ctypes.byref(weights),
                       _dev_ptr(x, torch.float32, "x"), x.shape[0],
                       _dev_ptr(idx, torch.int32, "idx"), _dev_ptr(w, torch.float32, "w"),
                       _dev_ptr(off, torch.int32, "off"), _dev_ptr(perm, torch.int32, "perm"),
                       _dev_ptr(pos, torch.int32, "pos"), _dev_ptr(y, torch.float32, "y"),
                       _dev_ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    _check("moe_ffn", st)


def layer(desc: MoeDesc, weights: MoeWeights, x, logits, bias, y, ws, stream=None):
    st = lib().moe_layer(ctypes.byref(desc), ctypes.byref(weights),
                         _dev_ptr(x, torch.float32, "x"), _dev_ptr(logits, torch.float32, "logits"),
                         _dev_ptr(bias, torch.float32, "bias"), x.shape[0],
                         _dev_ptr(y, torch.float32, "y"), _dev_ptr(ws, torch.uint8, "ws"),
                         ws.numel(), _stream(stream))
    _check("moe_layer", st)


def layer_from_x(desc: MoeDesc, weights: MoeWeights, w_router, x, bias, logits, y, ws,
                 stream=None):
    """moe_layer_from_x: router logits from x (written to ``logits``), then the
    layer on them; on the fused decode path the logits GEMM runs inside the
    decode kernel."""
    st = lib().moe_layer_from_x(ctypes.byref(desc), ctypes.byref(weights),
                                _dev_ptr(w_router, torch.float32, "w_router"),
                                _dev_ptr(x, torch.float32, "x"),
                                _dev_ptr(bias, torch.float32, "bias"), x.shape[0],
                                _dev_ptr(logits, torch.float32, "logits"),
                                _dev_ptr(y, torch.float32, "y"), _dev_ptr(ws, torch.uint8, "ws"),
                                ws.numel(), _stream(stream))
    _check("moe_layer_from_x", st)


def layer_timed(desc: MoeDesc, weights: MoeWeights, x, logits, bias, y, ws, events,
                stream=None):
    """moe_layer with ``events`` (torch.cuda.Event list) recorded between stages:
    events[0] before the first stage, events[i] after stage i-1."""
    for ev in events:  # torch creates the CUDA event lazily, on its first record
        if not ev.cuda_event:
            ev.record()
    handles = (_vp * len(events))(*[ev.cuda_event for ev in events])
    st = lib().moe_layer_timed(ctypes.byref(desc), ctypes.byref(weights),
                               _dev_ptr(x, torch.float32, "x"),
                               _dev_ptr(logits, torch.float32, "logits"),
                               _dev_ptr(bias, torch.float32, "bias"), x.shape[0],
                               _dev_ptr(y, torch.float32, "y"), _dev_ptr(ws, torch.uint8, "ws"),
                               ws.numel(), _stream(stream), handles, len(events))
    _check("moe_layer_timed", st)


def layer_experts(desc: MoeDesc, weights: MoeWeights, x, logits, bias, y, ws, begin: int,
                  end: int, with_shared: bool, stream=None):
    """moe_layer_experts: the layer restricted to routed experts [begin, end) and,
    if with_shared, the shared expert (one rank's share of an expert-parallel
    split; the ranks' outputs sum to the layer)."""
    st = lib().moe_layer_experts(ctypes.byref(desc), ctypes.byref(weights),
                                 _dev_ptr(x, torch.float32, "x"),
                                 _dev_ptr(logits, torch.float32, "logits"),
                                 _dev_ptr(bias, torch.float32, "bias"), x.shape[0], begin, end,
                                 1 if with_shared else 0, _dev_ptr(y, torch.float32, "y"),
                                 _dev_ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    _check("moe_layer_experts", st)


def ffn_experts(desc: MoeDesc, weights: MoeWeights, x, idx, w, off, perm, pos, y, ws,
                begin: int, end: int, with_shared: bool, stream=None):
    """moe_ffn_experts: moe_ffn restricted like layer_experts."""
    st = lib().moe_ffn_experts(ctypes.byref(desc), ctypes.byref(weights),
                               _dev_ptr(x, torch.float32, "x"), x.shape[0],
                               _dev_ptr(idx, torch.int32, "idx"), _dev_ptr(w, torch.float32, "w"),
                               _dev_ptr(off, torch.int32, "off"),
                               _dev_ptr(perm, torch.int32, "perm"),
                               _dev_ptr(pos, torch.int32, "pos"), begin, end,
                               1 if with_shared else 0, _dev_ptr(y, torch.float32, "y"),
                               _dev_ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    _check("moe_ffn_experts", st)


def layer_noalloc(desc: MoeDesc, weights: MoeWeights, x, logits, bias, y, stream=None):
    """moe_layer_noalloc: the layer without a workspace, for callers that cannot
    allocate device memory; scratch comes from the library's fixed 16 MiB device
    array (calls on one device must not overlap).  Its device error word is read
    (and cleared) by check_device_error(None)."""
    st = lib().moe_layer_noalloc(ctypes.byref(desc), ctypes.byref(weights),
                                 _dev_ptr(x, torch.float32, "x"),
                                 _dev_ptr(logits, torch.float32, "logits"),
                                 _dev_ptr(bias, torch.float32, "bias"), x.shape[0],
                                 _dev_ptr(y, torch.float32, "y"), _stream(stream))
    _check("moe_layer_noalloc", st)


NOALLOC_SCRATCH_BYTES = 16 << 20


def _host_ptr(t, name="tensor"):
    if t.is_cuda:
        raise ValueError(f"{name} must be host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _i32_host(a):
    """A host int32 array (numpy or CPU tensor) as (keep-alive object, pointer, n)."""
    import numpy as np

    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32).reshape(-1))
    return arr, arr.ctypes.data, int(arr.size)


class ExpertCache:
    """moe_cache_*: an HBM cache of expert slots over host-resident routed experts.

    ``host_layers``: one MoeWeights per layer whose gate/up/down point at pinned
    host planes; ``arena``: MoeWeights whose gate/up/down point at device planes
    of ``n_slots`` experts; ``slot_table``: device int32 [n_layers, E].  With
    ``policy_only`` the cache does no device work (plan / slot / stats only), and
    the pointers are not dereferenced."""

    def __init__(self, desc: MoeDesc, host_layers, arena: MoeWeights, n_slots: int,
                 slot_table_ptr: int, policy_only: bool = False):
        arr = (MoeWeights * len(host_layers))(*host_layers)
        h = ctypes.c_void_p()
        st = lib().moe_cache_create(ctypes.byref(desc), len(host_layers), arr, ctypes.byref(arena),
                                    n_slots, slot_table_ptr,
                                    CACHE_POLICY_ONLY if policy_only else 0, ctypes.byref(h))
        _check("moe_cache_create", st)
        self._h = h
        self._keep = (arr, arena)
        self.n_slots = n_slots

    def close(self):
        if self._h:
            lib().moe_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def ensure(self, layer: int, experts, stream=None):
        arr, ptr, n = _i32_host(experts)
        _check("moe_cache_ensure", lib().moe_cache_ensure(self._h, layer, ptr, n, _stream(stream)))

    def prefetch(self, layer: int, experts, stream=None):
        arr, ptr, n = _i32_host(experts)
        _check("moe_cache_prefetch", lib().moe_cache_prefetch(self._h, layer, ptr, n,
                                                              _stream(stream)))

    def plan(self, layer: int, experts, prefetch: bool = False):
        """Policy step only: returns [(expert, slot, evicted layer*E+expert or -1)]."""
        import numpy as np

        arr, ptr, n = _i32_host(experts)
        m = max(n, 1)
        loaded = np.zeros(m, np.int32)
        slots = np.zeros(m, np.int32)
        evicted = np.zeros(m, np.int64)
        cnt = _u32(0)
        _check("moe_cache_plan", lib().moe_cache_plan(
            self._h, layer, ptr, n, 1 if prefetch else 0, loaded.ctypes.data, slots.ctypes.data,
            evicted.ctypes.data, ctypes.byref(cnt)))
        return [(int(loaded[i]), int(slots[i]), int(evicted[i])) for i in range(cnt.value)]

    def slot(self, layer: int, expert: int) -> int:
        return int(lib().moe_cache_slot(self._h, layer, expert))

    def stats(self) -> dict:
        out = MoeCacheStats()
        _check("moe_cache_get_stats", lib().moe_cache_get_stats(self._h, ctypes.byref(out)))
        return {n: int(getattr(out, n)) for n, _ in MoeCacheStats._fields_}


def stream_layer(cache: ExpertCache, layer: int, desc: MoeDesc, shared: MoeWeights, x, logits,
                 bias, y, ws, next_logits=None, next_bias=None, stream=None,
                 prefetch_stream=None):
    """moe_stream_layer: route, make the picks resident in the cache, run the layer
    on the slot weights; with next_logits, prefetch the next layer's picks."""
    st = lib().moe_stream_layer(cache.handle, layer, ctypes.byref(desc), ctypes.byref(shared),
                                _dev_ptr(x, torch.float32, "x"),
                                _dev_ptr(logits, torch.float32, "logits"),
                                _dev_ptr(bias, torch.float32, "bias"), x.shape[0],
                                _dev_ptr(next_logits, torch.float32, "next_logits"),
                                _dev_ptr(next_bias, torch.float32, "next_bias"),
                                _dev_ptr(y, torch.float32, "y"), _dev_ptr(ws, torch.uint8, "ws"),
                                ws.numel(), _stream(stream), _stream(prefetch_stream))
    _check("moe_stream_layer", st)


def layer_path(desc: MoeDesc, T: int) -> str:
    return lib().moe_layer_path(ctypes.byref(desc), T).decode()


def tc_min_rows(desc: MoeDesc, T: int):
    """Experts with more rows than this run on the tensor cores; None: no tensor path."""
    v = lib().moe_tc_min_rows(ctypes.byref(desc), T)
    return None if v < 0 else v


def stage_names(desc: MoeDesc, T: int) -> list:
    names = []
    while True:
        n = lib().moe_layer_stage_name(ctypes.byref(desc), T, len(names))
        if n is None:
            return names
        names.append(n.decode())


def check_device_error(ws, stream=None) -> int:
    """Returns the moe_status of the workspace's device error word (and clears
    it; after a timeout also the workspace's counters).  ws=None: the static
    scratch of layer_noalloc on the current device."""
    if ws is None:
        return int(lib().moe_check_device_error(None, 0, _stream(stream)))
    return int(lib().moe_check_device_error(_dev_ptr(ws, torch.uint8, "ws"), ws.numel(),
                                            _stream(stream)))


# ------------------------------------------------------------------ convenience
@dataclass
class LayerOutput:
    y: torch.Tensor
    idx: torch.Tensor
    w: torch.Tensor
    off: torch.Tensor
    perm: torch.Tensor
    pos: torch.Tensor
    xq: torch.Tensor
    xs: torch.Tensor
    hq: torch.Tensor
    hs: torch.Tensor
    tap_gu: Optional[torch.Tensor]
    tap_dn: Optional[torch.Tensor]


class Layer:
    """One routed-MoE layer resident on a device: weights, descriptor, workspace.

    ``tensors`` holds the planar weights: ``gate_q`` [E,f,d] (int8, or uint8 2-bit
    codes [E,f,d/4]), ``gate_s`` [E,f,d/32] fp16, likewise ``up_*``, ``down_q``
    [E,d,f(/4)], ``down_s`` [E,d,f/32], and the shared expert as ``s_gate_q`` ...
    """

    def __init__(self, n_expert, top_k, d, f, f_shared, routed_fmt, s, tensors: dict,
                 device=None, score=SCORE_SIGMOID):
        self.n_expert, self.top_k, self.d, self.f = n_expert, top_k, d, f
        self.f_shared, self.routed_fmt, self.s = f_shared, routed_fmt, float(s)
        self.score = score
        self.tensors = tensors
        self.device = device or tensors["gate_q"].device
        self.weights = MoeWeights()
        names = ["gate", "up", "down"] + (["s_gate", "s_up", "s_down"] if f_shared else [])
        for n in names:
            q, sc = tensors[n + "_q"], tensors[n + "_s"]
            setattr(self.weights, n, MoeMat(_dev_ptr(q, None, n + "_q"),
                                           _dev_ptr(sc, torch.float16, n + "_s")))
        self._ws = {}

    @classmethod
    def from_host(cls, spec, experts: dict, shared: Optional[dict], device):
        """Stack per-expert host arrays (numpy, planar) into device tensors."""
        import numpy as np

        t = {}
        for name in ("gate", "up", "down"):
            q = np.stack([experts[e][name + "_q"] for e in range(spec.E)])
            sc = np.stack([np.asarray(experts[e][name + "_s"]).view(np.float16)
                           for e in range(spec.E)])
            t[name + "_q"] = torch.from_numpy(q).to(device)
            t[name + "_s"] = torch.from_numpy(sc).to(device)
            if spec.f_shared:
                t["s_" + name + "_q"] = torch.from_numpy(np.ascontiguousarray(
                    shared[name + "_q"])).to(device)
                t["s_" + name + "_s"] = torch.from_numpy(np.ascontiguousarray(
                    np.asarray(shared[name + "_s"]).view(np.float16))).to(device)
        return cls(spec.E, spec.k, spec.d, spec.f, spec.f_shared, spec.fmt, spec.s, t, device)

    def desc(self, flags=0) -> MoeDesc:
        return make_desc(self.n_expert, self.top_k, self.d, self.f, self.f_shared,
                         self.routed_fmt, self.s, flags, self.score)

    def workspace(self, T: int, flags=0) -> torch.Tensor:
        key = (T, flags & FLAG_DEBUG_TAPS)
        if key not in self._ws:
            n = workspace_size(self.desc(flags), T)
            self._ws[key] = torch.zeros(max(n, 256), dtype=torch.uint8, device=self.device)
        return self._ws[key]

    def views(self, ws: torch.Tensor, T: int, flags=0) -> dict:
        """Typed views of the workspace regions (for taps and tests)."""
        L = workspace_layout(self.desc(flags), T)
        R = T * self.top_k
        slots = R + (T if self.f_shared else 0)
        fmax = max(self.f, self.f_shared)

        def v(off, n, dtype, shape):
            nbytes = n * torch.tensor([], dtype=dtype).element_size()
            return ws[off:off + nbytes].view(dtype).view(shape)

        out = dict(
            idx=v(L.idx, R, torch.int32, (T, self.top_k)), w=v(L.w, R, torch.float32, (T, self.top_k)),
            off=v(L.off, self.n_expert + 1, torch.int32, (self.n_expert + 1,)),
            perm=v(L.perm, R, torch.int32, (R,)), pos=v(L.pos, R, torch.int32, (R,)),
            xq=v(L.xq, T * self.d, torch.int8, (T, self.d)),
            xs=v(L.xs, T * self.d // 32, torch.float32, (T, self.d // 32)),
            hq=v(L.hq, slots * fmax, torch.int8, (slots, fmax)),
            hs=v(L.hs, slots * fmax // 32, torch.float32, (slots, fmax // 32)),
            tap_gu=None, tap_dn=None)
        if flags & FLAG_DEBUG_TAPS:
            nt = L.n_tap
            out["tap_gu"] = v(L.tap_gu, slots * 2 * nt * (self.d // 32), torch.int32,
                              (slots, 2, nt, self.d // 32))
            out["tap_dn"] = v(L.tap_dn, slots * nt * (fmax // 32), torch.int32,
                              (slots, nt, fmax // 32))
        return out

    def forward(self, x: torch.Tensor, logits: torch.Tensor, bias: torch.Tensor,
                taps: bool = False, flags: int = 0, y: Optional[torch.Tensor] = None,
                stream=None) -> LayerOutput:
        flags = flags | (FLAG_DEBUG_TAPS if taps else 0)
        T = x.shape[0]
        ws = self.workspace(T, flags)
        if y is None:
            y = torch.empty((T, self.d), dtype=torch.float32, device=self.device)
        layer(self.desc(flags), self.weights, x, logits, bias, y, ws, stream)
        v = self.views(ws, T, flags)
        return LayerOutput(y=y, **v)

    def forward_from_x(self, x: torch.Tensor, w_router: torch.Tensor, bias: torch.Tensor,
                       logits: torch.Tensor, taps: bool = False, flags: int = 0,
                       y: Optional[torch.Tensor] = None, stream=None) -> LayerOutput:
        """moe_layer_from_x: the router logits of x (written to ``logits``
        [T][E]) and the layer on them, in one call."""
        flags = flags | (FLAG_DEBUG_TAPS if taps else 0)
        T = x.shape[0]
        ws = self.workspace(T, flags)
        if y is None:
            y = torch.empty((T, self.d), dtype=torch.float32, device=self.device)
        layer_from_x(self.desc(flags), self.weights, w_router, x, bias, logits, y, ws, stream)
        v = self.views(ws, T, flags)
        return LayerOutput(y=y, **v)
