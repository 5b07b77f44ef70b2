"""ctypes front end of the CPU oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg (and its ``--impl reference`` arm) may import this
module.  The product library never loads it and has no CPU fallback.

The arithmetic lives in C; this file only marshals numpy arrays.  Function
names mirror the C entry points; see ``oracle.h`` for the definitions and the
page citations.  Parity status per function: every function is pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_HERE, "liboracle.so")

FMT_Q8_0 = 0
FMT_Q2S = 1
FMT_E2M1 = 2
SCORE_SIGMOID = 0
SCORE_SQRT_SOFTPLUS = 1

_lib = None
_p = ctypes.c_void_p
_u32 = ctypes.c_uint32
_i32 = ctypes.c_int32


class _Expert(ctypes.Structure):
    _fields_ = [("gate_q", _p), ("gate_s", _p), ("up_q", _p), ("up_s", _p),
                ("down_q", _p), ("down_s", _p)]


class _Desc(ctypes.Structure):
    _fields_ = [("n_expert", _u32), ("top_k", _u32), ("d", _u32), ("f", _u32),
                ("f_shared", _u32), ("routed_fmt", _i32), ("s", ctypes.c_float),
                ("score_fn", _i32)]


class _Out(ctypes.Structure):
    _fields_ = [(n, _p) for n in ("idx", "w", "off", "perm", "pos", "xq", "xs", "hq_r",
                                  "hs_r", "hq_s", "hs_s", "y")]


def load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} missing: run __graft_entry__.build()")
        lib = ctypes.CDLL(LIB)
        lib.ora_spec_exp.restype = ctypes.c_float
        lib.ora_spec_exp.argtypes = [ctypes.c_float]
        lib.ora_spec_exp_n.argtypes = [_u32, _p, _p]
        lib.ora_f16_to_f64.restype = ctypes.c_double
        lib.ora_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.ora_score.argtypes = [_u32, _p, _p, _p, _p]
        lib.ora_spec_log1p.restype = ctypes.c_float
        lib.ora_spec_log1p.argtypes = [ctypes.c_float]
        lib.ora_sqrt_softplus.restype = ctypes.c_float
        lib.ora_sqrt_softplus.argtypes = [ctypes.c_float]
        lib.ora_router_logits.argtypes = [_u32, _u32, _u32, _p, _p, _p]
        lib.ora_score_fn.argtypes = [_i32, _u32, _p, _p, _p, _p]
        lib.ora_route_fn.argtypes = [_i32, _u32, _u32, _u32, ctypes.c_float, _p, _p, _p, _p]
        lib.ora_topk.argtypes = [_u32, _u32, _p, _p]
        lib.ora_route.argtypes = [_u32, _u32, _u32, ctypes.c_float, _p, _p, _p, _p]
        lib.ora_permute.argtypes = [_u32, _u32, _u32, _p, _p, _p, _p]
        lib.ora_quantize.argtypes = [_u32, _p, _p, _p]
        lib.ora_decode_q2.argtypes = [_u32, _p, _p]
        lib.ora_decode_e2m1.argtypes = [_u32, _p, _p]
        lib.ora_block_dots.argtypes = [_i32, _u32, _p, _p, _p]
        lib.ora_matvec.argtypes = [_i32, _u32, _u32, _p, _p, _p, _p, _p]
        lib.ora_expert_row.argtypes = [_i32, _u32, _u32, ctypes.POINTER(_Expert), _p, _p, _p,
                                       _p, _p]
        lib.ora_expert_row.restype = ctypes.c_int
        lib.ora_layer.argtypes = [ctypes.POINTER(_Desc), ctypes.POINTER(_Expert),
                                  ctypes.POINTER(_Expert), _u32, _p, _p, _p, _p,
                                  ctypes.POINTER(_Out)]
        lib.ora_layer.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------- step functions
def spec_exp(x) -> np.ndarray:
    x = _c(np.asarray(x, np.float32).ravel(), np.float32)
    out = np.empty_like(x)
    load().ora_spec_exp_n(x.size, _ptr(x), _ptr(out))
    return out


def f16_to_f64(bits: int) -> float:
    return float(load().ora_f16_to_f64(int(bits)))


def score(logit, bias):
    logit = _c(logit, np.float32)
    bias = _c(bias, np.float32)
    E = logit.size
    sigma = np.empty(E, np.float32)
    c = np.empty(E, np.float32)
    load().ora_score(E, _ptr(logit), _ptr(bias), _ptr(sigma), _ptr(c))
    return sigma, c


def spec_log1p(y) -> np.ndarray:
    lib = load()
    y = np.asarray(y, np.float32).ravel()
    return np.array([lib.ora_spec_log1p(float(v)) for v in y], np.float32)


def sqrt_softplus(logit) -> np.ndarray:
    lib = load()
    logit = np.asarray(logit, np.float32).ravel()
    return np.array([lib.ora_sqrt_softplus(float(v)) for v in logit], np.float32)


def router_logits(x, w_r) -> np.ndarray:
    """logits[T][E] = x[T][d] . w_r[E][d]^T: exact products summed in fp64,
    rounded once to fp32."""
    x = _c(x, np.float32)
    w_r = _c(w_r, np.float32)
    T, d = x.shape
    E = w_r.shape[0]
    out = np.empty((T, E), np.float32)
    load().ora_router_logits(T, E, d, _ptr(x), _ptr(w_r), _ptr(out))
    return out


def score_fn(fn: int, logit, bias):
    logit = _c(logit, np.float32)
    bias = _c(bias, np.float32)
    E = logit.size
    p = np.empty(E, np.float32)
    c = np.empty(E, np.float32)
    load().ora_score_fn(int(fn), E, _ptr(logit), _ptr(bias), _ptr(p), _ptr(c))
    return p, c


def topk(c, k: int) -> np.ndarray:
    c = _c(c, np.float32)
    idx = np.empty(k, np.int32)
    load().ora_topk(c.size, k, _ptr(c), _ptr(idx))
    return idx


def route(logits, bias, k: int, s: float, score: int = SCORE_SIGMOID):
    logits = _c(logits, np.float32)
    bias = _c(bias, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    load().ora_route_fn(int(score), T, E, k, float(s), _ptr(logits), _ptr(bias), _ptr(idx),
                        _ptr(w))
    return idx, w


def permute(idx, E: int):
    idx = _c(idx, np.int32)
    T, k = idx.shape
    off = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    pos = np.empty(T * k, np.int32)
    load().ora_permute(T, E, k, _ptr(idx), _ptr(off), _ptr(perm), _ptr(pos))
    return off, perm, pos


def quantize(x):
    x = _c(x, np.float32).ravel()
    q = np.empty(x.size, np.int8)
    sc = np.empty(x.size // 32, np.float32)
    load().ora_quantize(x.size, _ptr(x), _ptr(q), _ptr(sc))
    return q, sc


def decode_q2(codes, K: int) -> np.ndarray:
    codes = _c(codes, np.uint8)
    out = np.empty(K, np.int8)
    load().ora_decode_q2(K, _ptr(codes), _ptr(out))
    return out


def decode_e2m1(codes, K: int) -> np.ndarray:
    """4-bit e2m1 codes (two a byte, low nibble first) -> int8 TWICE the value."""
    codes = _c(codes, np.uint8)
    out = np.empty(K, np.int8)
    load().ora_decode_e2m1(K, _ptr(codes), _ptr(out))
    return out


def block_dots(fmt: int, K: int, wq_row, xq) -> np.ndarray:
    wq_row = _c(wq_row, np.int8 if fmt == FMT_Q8_0 else np.uint8)
    xq = _c(xq, np.int8)
    out = np.empty(K // 32, np.int32)
    load().ora_block_dots(fmt, K, _ptr(wq_row), _ptr(xq), _ptr(out))
    return out


def matvec(fmt: int, wq, ws, xq, xs) -> np.ndarray:
    wq = _c(wq, np.int8 if fmt == FMT_Q8_0 else np.uint8)
    ws = _c(np.asarray(ws).view(np.uint16) if np.asarray(ws).dtype == np.float16 else ws,
            np.uint16)
    rows = wq.shape[0]
    K = wq.shape[1] * {FMT_Q8_0: 1, FMT_Q2S: 4, FMT_E2M1: 2}[fmt]
    xq = _c(xq, np.int8)
    xs = _c(xs, np.float32)
    out = np.empty(rows, np.float64)
    load().ora_matvec(fmt, rows, K, _ptr(wq), _ptr(ws), _ptr(xq), _ptr(xs), _ptr(out))
    return out


def _expert_struct(ex: dict, keep: list) -> _Expert:
    st = _Expert()
    for name in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
        a = ex[name]
        if name.endswith("_s"):
            a = np.ascontiguousarray(np.asarray(a).view(np.uint16))
        else:
            a = np.ascontiguousarray(a)
        keep.append(a)
        setattr(st, name, a.ctypes.data)
    return st


def expert_row(fmt: int, d: int, width: int, ex: dict, xq, xs):
    keep = []
    st = _expert_struct(ex, keep)
    xq = _c(xq, np.int8)
    xs = _c(xs, np.float32)
    hq = np.empty(width, np.int8)
    hs = np.empty(width // 32, np.float32)
    o = np.empty(d, np.float64)
    rc = load().ora_expert_row(fmt, d, width, ctypes.byref(st), _ptr(xq), _ptr(xs), _ptr(hq),
                               _ptr(hs), _ptr(o))
    if rc != 0:
        raise RuntimeError(f"ora_expert_row failed: {rc}")
    return hq, hs, o


@dataclass
class LayerResult:
    idx: np.ndarray
    w: np.ndarray
    off: np.ndarray
    perm: np.ndarray
    pos: np.ndarray
    xq: np.ndarray
    xs: np.ndarray
    hq_r: np.ndarray
    hs_r: np.ndarray
    hq_s: np.ndarray
    hs_s: np.ndarray
    y: np.ndarray


def layer(E: int, k: int, d: int, f: int, f_shared: int, fmt: int, s: float,
          experts, shared, x, logits, bias, want=None, score: int = SCORE_SIGMOID) -> LayerResult:
    """Run the whole layer.  ``experts`` maps expert id -> dict of planar arrays
    (gate_q, gate_s, up_q, up_s, down_q, down_s); a missing id is allowed only if
    no wanted token selects it.  ``shared`` is such a dict, or None."""
    lib = load()
    x = _c(x, np.float32)
    logits = _c(logits, np.float32)
    bias = _c(bias, np.float32)
    T = x.shape[0]
    R = T * k
    keep = []
    arr = (_Expert * E)()
    for e in range(E):
        ex = experts.get(e) if isinstance(experts, dict) else experts[e]
        if ex is not None:
            arr[e] = _expert_struct(ex, keep)
    sh = _expert_struct(shared, keep) if (shared is not None and f_shared > 0) else _Expert()
    desc = _Desc(E, k, d, f, f_shared, fmt, float(s), int(score))
    res = LayerResult(
        idx=np.empty((T, k), np.int32), w=np.empty((T, k), np.float32),
        off=np.empty(E + 1, np.int32), perm=np.empty(R, np.int32), pos=np.empty(R, np.int32),
        xq=np.empty((T, d), np.int8), xs=np.empty((T, d // 32), np.float32),
        hq_r=np.zeros((R, f), np.int8), hs_r=np.zeros((R, f // 32), np.float32),
        hq_s=np.zeros((T, max(f_shared, 0)), np.int8),
        hs_s=np.zeros((T, max(f_shared, 0) // 32), np.float32),
        y=np.full((T, d), np.nan, np.float32))
    out = _Out()
    for name in _Out._fields_:
        n = name[0]
        a = getattr(res, n)
        setattr(out, n, a.ctypes.data if a.size else None)
    want_arr = None
    if want is not None:
        want_arr = np.zeros(T, np.uint8)
        want_arr[np.asarray(want, dtype=np.int64)] = 1
    rc = lib.ora_layer(ctypes.byref(desc), arr, ctypes.byref(sh), T, _ptr(x), _ptr(logits),
                       _ptr(bias), _ptr(want_arr), ctypes.byref(out))
    if rc != 0:
        raise RuntimeError(f"ora_layer failed: {rc}")
    return res
