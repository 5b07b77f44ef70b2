"""Independent numpy re-derivations used to pin the oracle (tests only).

Nothing here calls the oracle's arithmetic: weights are dequantised to fp64
matrices and the layer is recomputed with dense matmuls, a stable argsort and
a brute-force sort.  Agreement with the oracle (which uses scalar int32 block
dots, a scan-per-slot top-k and a counting sort) pins block indexing, scale
placement, gate/up order, the permutation and the combine order.
"""
from __future__ import annotations

import numpy as np


def f16_bits_to_f64(bits) -> np.ndarray:
    return np.asarray(bits).view(np.float16).astype(np.float64)


def decode_q2(codes: np.ndarray, K: int) -> np.ndarray:
    """Byte i//4, bits 2*(i%4) (LSB first); code c means 2c-3."""
    codes = np.asarray(codes, np.uint8)
    shifts = np.array([0, 2, 4, 6], np.uint8)
    c = (codes[..., :, None] >> shifts) & 3  # [..., K/4, 4]
    return (2 * c.reshape(codes.shape[:-1] + (K,)).astype(np.int16) - 3).astype(np.int8)


def decode_e2m1_value(codes: np.ndarray, K: int) -> np.ndarray:
    """4-bit e2m1 codes (byte i//2, bits 4*(i%2)) -> fp64 values, through
    numpy's float16 decoding: a normal code (e > 0) is the float16 with the
    same sign, exponent e - 1 (float16 field e + 14) and its mantissa bit as the
    top mantissa bit; a subnormal code (e == 0) is m * 0.5."""
    codes = np.asarray(codes, np.uint8)
    c = (codes[..., :, None] >> np.array([0, 4], np.uint8)) & 15
    c = c.reshape(codes.shape[:-1] + (K,)).astype(np.uint16)
    s, e, m = c >> 3, (c >> 1) & 3, c & 1
    bits = (s << 15) | ((e + 14) << 10) | (m << 9)
    v = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    sub = np.where(s == 1, -0.5, 0.5) * m
    return np.where(e == 0, sub, v)


def dequant(wq, ws, fmt: int, K: int) -> np.ndarray:
    """Planar weights -> fp64 matrix [rows, K]."""
    if fmt == 2:
        s = f16_bits_to_f64(np.asarray(ws).view(np.uint16))
        return decode_e2m1_value(wq, K) * np.repeat(s, 32, axis=1)
    q = decode_q2(wq, K) if fmt == 1 else np.asarray(wq, np.int8)
    s = f16_bits_to_f64(np.asarray(ws).view(np.uint16))  # [rows, K/32]
    return q.astype(np.float64) * np.repeat(s, 32, axis=1)


def round_half_away(v: np.ndarray) -> np.ndarray:
    v64 = np.asarray(v, np.float64)
    return np.sign(v64) * np.floor(np.abs(v64) + 0.5)


def quantize(x) -> tuple[np.ndarray, np.ndarray]:
    """Per 32-block: scale = max|x|/127 (fp32 division), q = round_half_away(x/scale)."""
    x = np.asarray(x, np.float32).reshape(-1, 32)
    a = np.abs(x).max(axis=1)
    sx = (a / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = (x / sx[:, None]).astype(np.float32)
    q = np.clip(round_half_away(quot), -127, 127)
    q[sx == 0] = 0
    return q.astype(np.int8).ravel(), sx


def sigmoid64(v):
    return 1.0 / (1.0 + np.exp(-np.asarray(v, np.float64)))


def expert_ffn(ex: dict, fmt: int, d: int, width: int, xq, xs):
    """Dense fp64 FFN of one expert on a quantised activation row.
    Returns (hq, hs, o)."""
    xd = np.asarray(xq, np.float64) * np.repeat(np.asarray(xs, np.float64), 32)
    Wg = dequant(ex["gate_q"], ex["gate_s"], fmt, d)
    Wu = dequant(ex["up_q"], ex["up_s"], fmt, d)
    g = Wg @ xd
    u = Wu @ xd
    h = (g * sigmoid64(g) * u).astype(np.float32)
    hq, hs = quantize(h)
    hd = hq.astype(np.float64) * np.repeat(hs.astype(np.float64), 32)
    Wd = dequant(ex["down_q"], ex["down_s"], fmt, width)
    return hq, hs, Wd @ hd


def brute_topk(c: np.ndarray, k: int) -> np.ndarray:
    """Full sort by (c descending, index ascending)."""
    order = sorted(range(len(c)), key=lambda i: (-float(c[i]), i))
    return np.array(order[:k], np.int32)


def stable_permutation(idx: np.ndarray, E: int):
    flat = np.asarray(idx, np.int64).ravel()
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    counts = np.bincount(flat, minlength=E)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    pos = np.empty_like(perm)
    pos[perm] = np.arange(perm.size, dtype=np.int32)
    return off, perm, pos


def sqrt_softplus64(v):
    v = np.asarray(v, np.float64)
    return np.sqrt(np.maximum(v, 0.0) + np.log1p(np.exp(-np.abs(v))))


def layer(E, k, d, f, f_shared, fmt, s, experts, shared, x, idx, logits, score=0):
    """Dense fp64 layer given the selected indices; returns y [T, d] (fp64).
    score: 0 sigmoid, 1 sqrt(softplus) (the routing weights' p)."""
    T = x.shape[0]
    y = np.zeros((T, d), np.float64)
    for t in range(T):
        xq, xs = quantize(x[t])
        acc = np.zeros(d, np.float64)
        if f_shared > 0:
            acc += expert_ffn(shared, 0, d, f_shared, xq, xs)[2]
        sg = (sqrt_softplus64 if score == 1 else sigmoid64)(logits[t, idx[t]])
        w = s * sg / sg.sum()
        for j in range(k):
            acc += w[j] * expert_ffn(experts[int(idx[t, j])], fmt, d, f, xq, xs)[2]
        y[t] = acc
    return y


def check_permutation(idx, off, perm, pos, E):
    """Invariants of the stable expert permutation; returns a list of failures."""
    flat = np.asarray(idx).ravel()
    R = flat.size
    bad = []
    if off[0] != 0 or off[E] != R:
        bad.append("off endpoints")
    if np.any(np.diff(off) < 0):
        bad.append("off not monotone")
    if not np.array_equal(np.diff(off), np.bincount(flat, minlength=E)[:E]):
        bad.append("counts differ from histogram")
    if not np.array_equal(np.sort(perm), np.arange(R)):
        bad.append("perm not a bijection")
    if not np.array_equal(pos[perm], np.arange(R)):
        bad.append("pos is not the inverse of perm")
    for e in range(E):
        seg = perm[off[e]:off[e + 1]]
        if np.any(flat[seg] != e):
            bad.append(f"segment {e} holds rows of another expert")
            break
        if np.any(np.diff(seg) <= 0):
            bad.append(f"segment {e} not in (token, slot) order")
            break
    return bad
