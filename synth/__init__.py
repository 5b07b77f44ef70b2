"""Seeded synthetic inputs for the routed-MoE layer (tests and bench only).

Everything here is a pure function of (seed, stream, index); the counter-based
generator is defined in ``synth.h``.  This module draws logits, bias,
activations and quantised expert weights in the planar layout the layer uses
(an int8 or 2-bit code plane plus an fp16 scale plane per 32-element block).
It performs none of the layer's arithmetic, so the CPU oracle and the CUDA
library can both consume its bytes while sharing no code with each other.

Workload recipe (stand-ins for the GLM-5.2 / Hy3 MoE layers the pages run):
  logits  : N(0,1) per (token, expert), plus a per-layer Zipf popularity offset
            -beta * 1.1 * ln(rank_e) over a seeded rank permutation
  bias    : N(0, 0.1) per expert (0.1 read as the standard deviation)
  x       : N(0,1) per (token, hidden)
  weights : int8 uniform on [-127, 127] (or uniform 2-bit codes, or uniform
            4-bit e2m1 codes), fp16 block scale (0.5 + U[0,1)) / (m * sqrt(K))
            with m = 127, 3 or 6, the largest magnitude the codes stand for
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_HERE, "libsynth.so")
DEV_LIB = os.path.join(_HERE, "libsynth_dev.so")

FMT_Q8_0 = 0
FMT_Q2S = 1
FMT_E2M1 = 2

# stream ids: token-level streams use the token seed, layer-level ones the layer seed
STREAM_LOGITS = 0
STREAM_BIAS = 1
STREAM_X = 2
STREAM_ZIPF = 3
STREAM_ROUTER = 4  # router weights W_r [E][d]
STREAM_WEIGHTS = 16  # + 8 * expert + matrix (expert == E is the shared expert)
MATS = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")

_host = None
_dev = None


def _load_host():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            raise RuntimeError(f"{HOST_LIB} missing: run __graft_entry__.build()")
        lib = ctypes.CDLL(HOST_LIB)
        u64, p = ctypes.c_uint64, ctypes.c_void_p
        lib.synth_draw.restype = u64
        lib.synth_draw.argtypes = [u64, u64, u64]
        lib.synth_int8.argtypes = [u64, u64, u64, u64, p]
        lib.synth_code2.argtypes = [u64, u64, u64, u64, p]
        lib.synth_scale_f16.argtypes = [u64, u64, u64, u64, ctypes.c_double, p]
        lib.synth_normal_f32.argtypes = [u64, u64, u64, u64, ctypes.c_double, ctypes.c_double, p]
        lib.synth_zipf_offset.argtypes = [u64, u64, ctypes.c_uint32, ctypes.c_double,
                                          ctypes.c_double, p]
        lib.synth_f64_to_f16.restype = ctypes.c_uint16
        lib.synth_f64_to_f16.argtypes = [ctypes.c_double]
        _host = lib
    return _host


def _load_dev():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_LIB):
            raise RuntimeError(f"{DEV_LIB} missing: run __graft_entry__.build()")
        lib = ctypes.CDLL(DEV_LIB)
        u64, p = ctypes.c_uint64, ctypes.c_void_p
        lib.synth_dev_int8.argtypes = [p, u64, u64, u64, u64, p]
        lib.synth_dev_code2.argtypes = [p, u64, u64, u64, u64, p]
        lib.synth_dev_scale_f16.argtypes = [p, u64, u64, u64, u64, ctypes.c_double, p]
        for fn in (lib.synth_dev_int8, lib.synth_dev_code2, lib.synth_dev_scale_f16):
            fn.restype = ctypes.c_int
        _dev = lib
    return _dev


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


# ---------------------------------------------------------------- raw streams
def draw(seed: int, stream: int, i: int) -> int:
    return int(_load_host().synth_draw(seed, stream, i))


def int8(seed: int, stream: int, n: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, np.int8)
    _load_host().synth_int8(seed, stream, first, n, _ptr(out))
    return out


def code2(seed: int, stream: int, n: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, np.uint8)
    _load_host().synth_code2(seed, stream, first, n, _ptr(out))
    return out


def scale_f16(seed: int, stream: int, n: int, denom: float, first: int = 0) -> np.ndarray:
    out = np.empty(n, np.uint16)
    _load_host().synth_scale_f16(seed, stream, first, n, float(denom), _ptr(out))
    return out.view(np.float16)


def normal(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0,
           first: int = 0) -> np.ndarray:
    out = np.empty(n, np.float32)
    _load_host().synth_normal_f32(seed, stream, first, n, float(mean), float(std), _ptr(out))
    return out


def zipf_offset(seed: int, stream: int, n_expert: int, beta: float, a: float = 1.1) -> np.ndarray:
    out = np.empty(n_expert, np.float32)
    _load_host().synth_zipf_offset(seed, stream, n_expert, float(beta), float(a), _ptr(out))
    return out


def f64_to_f16_bits(v: float) -> int:
    return int(_load_host().synth_f64_to_f16(float(v)))


# ---------------------------------------------------------------- layer specs
@dataclass(frozen=True)
class LayerSpec:
    """Shape of one routed-MoE layer."""
    name: str
    E: int           # routed experts
    k: int           # experts per token
    d: int           # hidden size
    f: int           # routed expert width
    f_shared: int    # shared expert width (0: no shared expert)
    fmt: int         # routed weight format: FMT_Q8_0, FMT_Q2S or FMT_E2M1
    s: float         # routing scale
    zipf_beta: float  # popularity-offset strength (0: none)
    layer_seed: int = 0
    score: int = 0    # logit scoring: 0 sigmoid, 1 sqrt(softplus)


TINY = LayerSpec("tiny", E=16, k=4, d=256, f=128, f_shared=0, fmt=FMT_Q8_0, s=1.0, zipf_beta=0.0)
GLM_LAYER = LayerSpec("e256_k8_d6144_f2048_q8", E=256, k=8, d=6144, f=2048, f_shared=2048,
                      fmt=FMT_Q8_0, s=2.5, zipf_beta=0.4)
Q2_LAYER = LayerSpec("e192_k8_d4096_f1536_q2", E=192, k=8, d=4096, f=1536, f_shared=1536,
                     fmt=FMT_Q2S, s=1.0, zipf_beta=0.4)
# the 2-bit layer's shape with 4-bit e2m1 routed experts (the same Hy3-sized
# layer in a format GB300's tensor cores take natively)
E2M1_LAYER = LayerSpec("e192_k8_d4096_f1536_e2m1", E=192, k=8, d=4096, f=1536, f_shared=1536,
                       fmt=FMT_E2M1, s=1.0, zipf_beta=0.4)

# Same per-token shapes as GLM_LAYER with 32 experts (1.3 GB of weights, 361 MB
# read per token): the small case that profiler captures run on.
# DeepSeek-style routing (sqrt(softplus) scoring, top-6, scale 1.5, 384 experts:
# "256 experts, 512 lines", section "The constant that always said 256") on the
# same expert shapes; no Zipf offset (its logits come from the router GEMM).
DS_LAYER = LayerSpec("e384_k6_d6144_f2048_q8_ds", E=384, k=6, d=6144, f=2048, f_shared=2048,
                     fmt=FMT_Q8_0, s=1.5, zipf_beta=0.0, score=1)

GLM_LAYER_E32 = LayerSpec("e32_k8_d6144_f2048_q8", E=32, k=8, d=6144, f=2048, f_shared=2048,
                          fmt=FMT_Q8_0, s=2.5, zipf_beta=0.4)
# 64 experts (2.4 GB): with T=128 an expert gets ~16 rows, as in a T=512 batch
# over 256 experts -- the small case for captures of the tensor-core path.
GLM_LAYER_E64 = LayerSpec("e64_k8_d6144_f2048_q8", E=64, k=8, d=6144, f=2048, f_shared=2048,
                          fmt=FMT_Q8_0, s=2.5, zipf_beta=0.4)

# workloads: (layer, tokens per step, token seeds)
WORKLOADS = {
    "tiny_t4": (TINY, 4, (0,)),
    "decode_t1": (GLM_LAYER, 1, tuple(range(100))),
    "batch_t16": (GLM_LAYER, 16, (0,)),
    "batch_t2": (GLM_LAYER, 2, (0,)),
    "prefill_t512": (GLM_LAYER, 512, (0,)),
    "q2_t64": (Q2_LAYER, 64, (0,)),
    "fp4_t64": (E2M1_LAYER, 64, (0,)),
    "profile_decode_t1": (GLM_LAYER_E32, 1, tuple(range(8))),
    "profile_batch_t16": (GLM_LAYER_E32, 16, (0,)),
    "profile_prefill_t512": (GLM_LAYER_E32, 512, (0,)),
    "profile_prefill_e64_t128": (GLM_LAYER_E64, 128, (0,)),
}


def weight_stream(expert: int, mat: str) -> int:
    return STREAM_WEIGHTS + 8 * expert + MATS.index(mat)


def expert_dims(spec: LayerSpec, expert: int):
    """(fmt, width, d) of a routed expert (expert < E) or of the shared one (expert == E)."""
    if expert == spec.E:
        return FMT_Q8_0, spec.f_shared, spec.d
    return spec.fmt, spec.f, spec.d


def scale_denom(fmt: int, K: int) -> float:
    return {FMT_Q8_0: 127.0, FMT_Q2S: 3.0, FMT_E2M1: 6.0}[fmt] * math.sqrt(K)


def matrix_shapes(fmt: int, rows: int, K: int):
    """(code-plane shape, scale-plane shape) of a [rows, K] matrix in planar layout."""
    qcols = {FMT_Q8_0: K, FMT_Q2S: K // 4, FMT_E2M1: K // 2}[fmt]
    return (rows, qcols), (rows, K // 32)


def expert_host(spec: LayerSpec, expert: int) -> dict:
    """Host arrays of one expert: gate/up [width, d], down [d, width]."""
    fmt, width, d = expert_dims(spec, expert)
    seed = spec.layer_seed
    out = {}
    for name, rows, K in (("gate", width, d), ("up", width, d), ("down", d, width)):
        qshape, sshape = matrix_shapes(fmt, rows, K)
        nq = qshape[0] * qshape[1]
        if fmt == FMT_Q8_0:
            q = int8(seed, weight_stream(expert, name + "_q"), nq)
        else:
            q = code2(seed, weight_stream(expert, name + "_q"), nq)
        sc = scale_f16(seed, weight_stream(expert, name + "_s"), sshape[0] * sshape[1],
                       scale_denom(fmt, K))
        out[name + "_q"] = q.reshape(qshape)
        out[name + "_s"] = sc.reshape(sshape)
    return out


def bias(spec: LayerSpec) -> np.ndarray:
    return normal(spec.layer_seed, STREAM_BIAS, spec.E, 0.0, 0.1)


def router_weights(spec: LayerSpec) -> np.ndarray:
    """Router weights W_r [E][d] fp32, N(0, 1/d): with x ~ N(0, 1) the logits
    x . W_r are ~N(0, 1), like the direct logits of token_inputs."""
    return normal(spec.layer_seed, STREAM_ROUTER, spec.E * spec.d, 0.0,
                  1.0 / float(np.sqrt(spec.d))).reshape(spec.E, spec.d)


def token_inputs(spec: LayerSpec, seed: int, T: int):
    """(logits [T,E] fp32, x [T,d] fp32) for one batch of T tokens."""
    logits = normal(seed, STREAM_LOGITS, T * spec.E).reshape(T, spec.E)
    if spec.zipf_beta > 0:
        off = zipf_offset(spec.layer_seed, STREAM_ZIPF, spec.E, spec.zipf_beta)
        logits = (logits + off[None, :]).astype(np.float32)
    x = normal(seed, STREAM_X, T * spec.d).reshape(T, spec.d)
    return np.ascontiguousarray(logits), np.ascontiguousarray(x)


# ---------------------------------------------------------------- device fill
def fill_layer_device(spec: LayerSpec, device="cuda"):
    """Allocate and fill all expert weights of ``spec`` in device memory.

    Returns a dict of torch tensors: ``gate_q`` [E, f, d(/4)], ``gate_s`` [E, f, d/32]
    (fp16), likewise ``up_*``, ``down_q`` [E, d, f(/4)], ``down_s`` [E, d, f/32], and
    the shared expert as ``s_gate_q`` ... (absent when f_shared == 0).
    """
    import torch

    lib = _load_dev()
    stream = torch.cuda.current_stream(device).cuda_stream
    seed = spec.layer_seed
    out = {}

    def fill(prefix, experts, fmt, width):
        for name, rows, K in (("gate", width, spec.d), ("up", width, spec.d),
                              ("down", spec.d, width)):
            qshape, sshape = matrix_shapes(fmt, rows, K)
            q = torch.empty((len(experts),) + qshape,
                            dtype=torch.int8 if fmt == FMT_Q8_0 else torch.uint8, device=device)
            sc = torch.empty((len(experts),) + sshape, dtype=torch.float16, device=device)
            nq = qshape[0] * qshape[1]
            ns = sshape[0] * sshape[1]
            for i, e in enumerate(experts):
                qp = ctypes.c_void_p(q.data_ptr() + i * nq)
                sp = ctypes.c_void_p(sc.data_ptr() + i * ns * 2)
                if fmt == FMT_Q8_0:
                    rc = lib.synth_dev_int8(qp, seed, weight_stream(e, name + "_q"), 0, nq,
                                            ctypes.c_void_p(stream))
                else:
                    rc = lib.synth_dev_code2(qp, seed, weight_stream(e, name + "_q"), 0, nq,
                                             ctypes.c_void_p(stream))
                if rc != 0:
                    raise RuntimeError(f"synth device fill failed: cuda error {rc}")
                rc = lib.synth_dev_scale_f16(sp, seed, weight_stream(e, name + "_s"), 0, ns,
                                             scale_denom(fmt, K), ctypes.c_void_p(stream))
                if rc != 0:
                    raise RuntimeError(f"synth device fill failed: cuda error {rc}")
            out[prefix + name + "_q"] = q
            out[prefix + name + "_s"] = sc

    fill("", list(range(spec.E)), spec.fmt, spec.f)
    if spec.f_shared > 0:
        fill("s_", [spec.E], FMT_Q8_0, spec.f_shared)
        for key in [k for k in out if k.startswith("s_")]:
            out[key] = out[key][0]
    return out
