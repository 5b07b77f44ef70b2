"""Shared machinery of the GPU parity tests: build a layer on the device from
the seeded generator, run it through the C ABI, run the CPU oracle on the same
bytes, and compare.

Bar (the layer's contract): bit-exact expert indices, offsets, permutation,
int8 activation codes + scales and int32 block dots; routing weights within
fp32 rounding; h codes within one step (rare, where fp32 summation order moves
h across a rounding boundary); y within 1e-3 normwise relative error per token.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
from routed_expert_decode_gb300 import moe

Y_TOL = 1e-3         # max_m |y_gpu - y_ora| / max_m |y_ora|, per token
W_RTOL = 4e-6        # fp32 routing weights vs the fp64 oracle
HQ_FLIP_FRAC = 1e-3  # fraction of h codes allowed to differ (by exactly one step)

_LAYERS = {}
_HOST = {}


def device_layer(spec: synth.LayerSpec, device) -> moe.Layer:
    key = (spec, str(device))
    if key not in _LAYERS:
        _LAYERS.clear()  # one resident layer at a time (full-size layers are ~10 GB)
        torch.cuda.empty_cache()
        t = synth.fill_layer_device(spec, device)
        torch.cuda.synchronize()
        _LAYERS[key] = moe.Layer(spec.E, spec.k, spec.d, spec.f, spec.f_shared, spec.fmt, spec.s,
                                 t, device, score=spec.score)
    return _LAYERS[key]


def host_expert(spec, e):
    key = (spec, e)
    if key not in _HOST:
        if len(_HOST) > 64:
            _HOST.clear()
        _HOST[key] = synth.expert_host(spec, e)
    return _HOST[key]


def run_case(spec, T, seed, device, sample=None, flags=0, check_taps=True, router=False):
    """Run one batch on the GPU and the oracle; assert parity; return a report.
    router=True: the logits come from the router GEMM x . W_r (moe_router_logits
    on the GPU, ora_router_logits on the CPU), which must agree bit for bit;
    router="fused": the same through moe_layer_from_x, which computes the logits
    and runs the layer in one call."""
    logits, x = synth.token_inputs(spec, seed, T)
    bias = synth.bias(spec)
    layer = device_layer(spec, device)
    taps = check_taps
    if router:
        w_r = synth.router_weights(spec)
        logits = oracle.router_logits(x, w_r)
        l_dev = torch.full((T, spec.E), float("nan"), dtype=torch.float32, device=device)
        w_dev, x_dev = torch.from_numpy(w_r).to(device), torch.from_numpy(x).to(device)
        if router == "fused":
            out = layer.forward_from_x(x_dev, w_dev, torch.from_numpy(bias).to(device), l_dev,
                                       taps=taps, flags=flags)
        else:
            moe.router_logits(layer.desc(), w_dev, x_dev, l_dev)
        torch.cuda.synchronize()
        assert np.array_equal(l_dev.cpu().numpy().view(np.uint32), logits.view(np.uint32)), \
            "router logits differ"
    if router != "fused":
        out = layer.forward(torch.from_numpy(x).to(device), torch.from_numpy(logits).to(device),
                            torch.from_numpy(bias).to(device), taps=taps, flags=flags)
    torch.cuda.synchronize()
    assert moe.check_device_error(layer.workspace(T, flags | (moe.FLAG_DEBUG_TAPS if taps else 0))) == 0

    # routing first (cheap for any T), then the oracle FFN on the sampled tokens
    if sample is None:
        sample = list(range(T))
    sample = sorted(set(int(t) for t in sample))
    r_idx, _ = oracle.route(logits, bias, spec.k, spec.s, score=spec.score)
    need = sorted(set(int(e) for t in sample for e in r_idx[t]))
    experts = {e: host_expert(spec, e) for e in need}
    shared = host_expert(spec, spec.E) if spec.f_shared else None
    ref = oracle.layer(spec.E, spec.k, spec.d, spec.f, spec.f_shared, spec.fmt, spec.s, experts,
                       shared, x, logits, bias, want=sample, score=spec.score)

    g = {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in vars(out).items()}
    R = T * spec.k
    # ---- bit-exact integer work
    assert np.array_equal(g["idx"], ref.idx), "expert indices differ"
    assert np.array_equal(g["off"], ref.off), "expert offsets differ"
    assert np.array_equal(g["perm"], ref.perm), "permutation differs"
    assert np.array_equal(g["pos"], ref.pos), "inverse permutation differs"
    assert np.array_equal(g["xq"], ref.xq), "int8 activations differ"
    assert np.array_equal(g["xs"], ref.xs), "activation scales differ"
    # ---- routing weights
    assert np.allclose(g["w"], ref.w, rtol=W_RTOL, atol=0), "routing weights differ"
    # ---- h codes of the sampled tokens' rows
    slots = [(int(ref.pos[t * spec.k + j]), t, int(ref.idx[t, j]), spec.f, False)
             for t in sample for j in range(spec.k)]
    if spec.f_shared:
        slots += [(R + t, t, spec.E, spec.f_shared, True) for t in sample]
    flips = 0
    total = 0
    for slot, t, e, width, is_shared in slots:
        ghq = g["hq"][slot, :width].astype(np.int32)
        rhq = (ref.hq_s[t] if is_shared else ref.hq_r[slot]).astype(np.int32)
        diff = np.abs(ghq - rhq)
        assert diff.max() <= 1, f"h codes differ by {diff.max()} in slot {slot}"
        flips += int((diff > 0).sum())
        total += width
    flip_frac = flips / max(total, 1)
    assert flip_frac <= HQ_FLIP_FRAC, f"h code flips {flip_frac:.2e}"
    # ---- int32 block dots (taps): gate/up exactly; down conditionally on the GPU's hq
    if taps:
        nt = 8
        for slot, t, e, width, is_shared in slots:
            ex = experts[e] if not is_shared else shared
            fmt = oracle.FMT_Q8_0 if is_shared else spec.fmt
            for j in range(nt):
                n = (j * width // nt + j) % width
                for mi, name in enumerate(("gate", "up")):
                    ref_dots = oracle.block_dots(fmt, spec.d, ex[name + "_q"][n], ref.xq[t])
                    assert np.array_equal(g["tap_gu"][slot, mi, j], ref_dots), \
                        f"{name} block dots differ (slot {slot}, feature {n})"
                m = (j * spec.d // nt + j) % spec.d
                ref_dn = oracle.block_dots(fmt, width, ex["down_q"][m], g["hq"][slot, :width])
                assert np.array_equal(g["tap_dn"][slot, j, :width // 32], ref_dn), \
                    f"down block dots differ (slot {slot}, output {m})"
    # ---- y
    y_err = []
    for t in sample:
        den = np.abs(ref.y[t]).max()
        y_err.append(float(np.abs(g["y"][t] - ref.y[t]).max() / den))
    assert max(y_err) <= Y_TOL, f"y normwise relative error {max(y_err):.3e}"
    return dict(max_y_err=max(y_err), hq_flip_frac=flip_frac, U=int((np.diff(ref.off) > 0).sum()))
