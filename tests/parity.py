"""Shared machinery of the GPU parity tests: build a layer on the device from
the seeded generator, run it through the C ABI, run the CPU oracle on the same
bytes, and compare.

Bar (the layer's contract): bit-exact expert indices, offsets, permutation,
int8 activation codes + scales and int32 block dots; routing weights within
fp32 rounding; h codes within one step (rare, where fp32 summation order moves
h across a rounding boundary); y within 1e-3 normwise relative error per token.
Elementwise, y is also checked within 1e-3 relative wherever |y| >= 1e-2 of the
token's max|y|, against the oracle's down projection and combine run on the
GPU's own h codes (a small output cannot hide under the normwise bound; a
one-step h-code flip, which the bar allows, moves small outputs by ~1e-2 of
their size, so the elementwise check is conditional on the h codes, like the
down-projection block dots).

Router logits computed from x (moe_router_logits, moe_layer_from_x) follow the
kernels' fixed fp32 summation order; the oracle's logit is the exact dot
rounded once.  They are compared within the fp32 error bound of that order,
and the routing and the layer are then checked conditionally on the GPU's own
logits (oracle.route on them must give the GPU's picks exactly).
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
Y_ELEM_FLOOR = 1e-2  # elementwise check where |y| >= this fraction of the token's max
Y_ELEM_TOL = 1e-3    # elementwise relative error above that floor, given the GPU's h codes
WS_FIXED_BYTES = 256 + 16384  # moe.h MOE_WS_FIXED_BYTES: error word + counters

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


def router_logit_bound(x, w_r):
    """fp32 error bound of the kernels' router order against the exact dot: a
    <= 32-long fma chain per lane and 1024-input segment, a 5-level tree, the
    segment totals added in order (one rounding each), plus half an ulp for the
    oracle's own rounding of the exact value."""
    d = x.shape[1]
    nseg = (d + 1023) // 1024
    mag = np.abs(x).astype(np.float64) @ np.abs(w_r).T.astype(np.float64)
    return (32 + 5 + nseg + 1) * 2.0 ** -24 * mag


def check_router_logits(x, w_r, l_gpu):
    """GPU logits within the bound of the oracle's (the dot rounded once)."""
    ref = oracle.router_logits(x, w_r).astype(np.float64)
    err = np.abs(l_gpu.astype(np.float64) - ref)
    bound = router_logit_bound(x, w_r)
    assert np.all(err <= bound + 1e-30), f"router logits off by {(err / (bound + 1e-30)).max():.2f}x the bound"
    return ref.astype(np.float32)


def poison_workspace(ws):
    """0xFF everywhere past the fixed head (error word + counters, which every
    call leaves zeroed): anything a kernel reads before writing turns into NaN
    floats, out-of-range indices and -1 codes."""
    ws[WS_FIXED_BYTES:].fill_(0xFF)


def run_case(spec, T, seed, device, sample=None, flags=0, check_taps=True, router=False,
             poison=False):
    """Run one batch on the GPU and the oracle; assert parity; return a report.
    router=True: the logits come from the router GEMM x . W_r (moe_router_logits
    on the GPU, ora_router_logits on the CPU), compared within the fp32 bound;
    router="fused": the same through moe_layer_from_x, which computes the logits
    and runs the layer in one call.  poison=True: the workspace is filled with
    0xFF past its fixed head before the call."""
    logits, x = synth.token_inputs(spec, seed, T)
    bias = synth.bias(spec)
    layer = device_layer(spec, device)
    taps = check_taps
    if poison:
        poison_workspace(layer.workspace(T, flags | (moe.FLAG_DEBUG_TAPS if taps else 0)))
    pick_diff = None
    if router:
        w_r = synth.router_weights(spec)
        l_dev = torch.full((T, spec.E), float("nan"), dtype=torch.float32, device=device)
        w_dev, x_dev = torch.from_numpy(w_r).to(device), torch.from_numpy(x).to(device)
        if router == "fused":
            out = layer.forward_from_x(x_dev, w_dev, torch.from_numpy(bias).to(device), l_dev,
                                       taps=taps, flags=flags)
        else:
            moe.router_logits(layer.desc(), w_dev, x_dev, l_dev)
        torch.cuda.synchronize()
        l_gpu = l_dev.cpu().numpy()
        l_ora = check_router_logits(x, w_r, l_gpu)
        # picks on the oracle's own logits, for the report (not a bar: a logit
        # one ulp apart can swap a near tie)
        i_ora, _ = oracle.route(l_ora, bias, spec.k, spec.s, score=spec.score)
        i_gpu, _ = oracle.route(l_gpu, bias, spec.k, spec.s, score=spec.score)
        pick_diff = int((np.sort(i_ora, axis=1) != np.sort(i_gpu, axis=1)).any(axis=1).sum())
        logits = l_gpu  # conditional parity from here on: the GPU's own logits
    if router != "fused":
        out = layer.forward(torch.from_numpy(x).to(device), torch.from_numpy(logits).to(device),
                            torch.from_numpy(bias).to(device), taps=taps, flags=flags)
    torch.cuda.synchronize()
    assert moe.check_device_error(layer.workspace(T, flags | (moe.FLAG_DEBUG_TAPS if taps else 0))) == 0
    g = {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in vars(out).items()}
    rep = compare_with_oracle(spec, T, x, logits, bias, g, sample=sample, taps=taps)
    if pick_diff is not None:
        rep["tokens_with_other_picks_on_oracle_logits"] = pick_diff
    return rep


def compare_with_oracle(spec, T, x, logits, bias, g, sample=None, taps=False):
    """The oracle layer on the same inputs against the GPU results `g` (numpy
    arrays named as in moe.LayerOutput: y, idx, w, off, perm, pos, xq, xs, hq,
    tap_gu, tap_dn); asserts the parity bar and returns a report."""
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
    flipped = set()  # sampled tokens with a one-step h flip in one of their rows
    for slot, t, e, width, is_shared in slots:
        ghq = g["hq"][slot, :width].astype(np.int32)
        rhq = (ref.hq_s[t] if is_shared else ref.hq_r[slot]).astype(np.int32)
        diff = np.abs(ghq - rhq)
        assert diff.max() <= 1, f"h codes differ by {diff.max()} in slot {slot}"
        flips += int((diff > 0).sum())
        total += width
        if diff.max() > 0:
            flipped.add(t)
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
    # ---- y: normwise per token (the bar) against the oracle's y for a token
    # whose h codes all equal the oracle's; for a token with a one-step h flip
    # (allowed above: the fp32 sums of g and u sit on a rounding boundary),
    # against y_c, the oracle's down projection (fp64 sums of the exact block
    # dots) and combine on the GPU's own h codes and scales -- at small widths
    # one flip alone moves y by ~1/(127 sqrt(f)) of its size.  Elementwise above
    # a floor, always against y_c.
    y_err, y_err_c, y_elem, y_elem_unc = [], [], [], []
    for t in sample:
        den = np.abs(ref.y[t]).max()
        err_t = float(np.abs(g["y"][t] - ref.y[t]).max() / den)
        big = np.abs(ref.y[t]) >= Y_ELEM_FLOOR * den
        rel = np.abs(g["y"][t][big] - ref.y[t][big]) / np.abs(ref.y[t][big])
        y_elem_unc.append(float(rel.max()) if rel.size else 0.0)
        yc = np.zeros(spec.d, np.float64)
        if spec.f_shared:
            yc += oracle.matvec(oracle.FMT_Q8_0, shared["down_q"], shared["down_s"],
                                g["hq"][R + t, :spec.f_shared], g["hs"][R + t, :spec.f_shared // 32])
        for j in range(spec.k):
            sl, e = int(ref.pos[t * spec.k + j]), int(ref.idx[t, j])
            yc += float(ref.w[t, j]) * oracle.matvec(spec.fmt, experts[e]["down_q"],
                                                     experts[e]["down_s"], g["hq"][sl, :spec.f],
                                                     g["hs"][sl, :spec.f // 32])
        bigc = np.abs(yc) >= Y_ELEM_FLOOR * np.abs(yc).max()
        relc = np.abs(g["y"][t][bigc] - yc[bigc]) / np.abs(yc[bigc])
        y_elem.append(float(relc.max()) if relc.size else 0.0)
        err_c = float(np.abs(g["y"][t] - yc).max() / np.abs(yc).max())
        y_err_c.append(err_c)
        assert (err_c if t in flipped else err_t) <= Y_TOL, \
            f"y normwise relative error {err_t:.3e} (token {t}; given the GPU's h codes {err_c:.3e})"
        y_err.append(err_t)
    assert max(y_elem) <= Y_ELEM_TOL, \
        f"y elementwise relative error {max(y_elem):.3e} (given the GPU's h codes)"
    return dict(max_y_err=max(y_err), max_y_err_given_h=max(y_err_c),
                max_y_elem_err_given_h=max(y_elem), max_y_elem_err=max(y_elem_unc),
                hq_flip_frac=flip_frac, tokens_with_flips=len(flipped),
                U=int((np.diff(ref.off) > 0).sum()))
