"""Expert-parallel split through the C ABI on one GB300 (pytest -m gpu).

The ranks of a split are emulated one after another on one GPU (each rank's
call is independent: no kernel waits on another rank).  Each rank runs
moe_layer_experts on its expert range -- on every path: the fused decode kernel
(T <= 2), the dp4a GEMV and the tensor cores -- optionally with weights that
hold only its own experts (an expert -> slot table whose other entries are
invalid, so a read of an unowned expert would fail the device check); the
partial outputs summed over the ranks must match the CPU oracle layer like
moe_layer itself (y within 1e-3 normwise), and moe_layer's y within the same
tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import Y_TOL, device_layer, host_expert
from routed_expert_decode_gb300 import moe
from routed_expert_decode_gb300.expert_parallel import ExpertParallel, expert_ranges

pytestmark = pytest.mark.gpu

ROUTED = ("gate", "up", "down")


def _spec(**kw):
    base = dict(name="ep", E=32, k=4, d=512, f=256, f_shared=256, fmt=0, s=2.5, zipf_beta=0.4)
    base.update(kw)
    return synth.LayerSpec(**base)


def _owned_weights(layer, lo, hi, dev):
    """The rank's weights: only experts [lo, hi) in slots 0..hi-lo-1; every
    other expert maps to slot hi-lo (out of range)."""
    n = hi - lo
    keep = {}
    w = moe.MoeWeights()
    for name in ROUTED:
        for sfx in ("_q", "_s"):
            keep[name + sfx] = layer.tensors[name + sfx][lo:hi].clone()
        setattr(w, name, moe.MoeMat(keep[name + "_q"].data_ptr(), keep[name + "_s"].data_ptr()))
    for name in ("s_gate", "s_up", "s_down"):
        setattr(w, name, getattr(layer.weights, name))
    table = np.full(layer.n_expert, n, np.int32)
    table[lo:hi] = np.arange(n)
    keep["table"] = torch.from_numpy(table).to(dev)
    w.expert_slot = keep["table"].data_ptr()
    w.n_slots = n
    return w, keep


def _oracle_y(spec, x, logits, bias, sample):
    idx, _ = oracle.route(logits, bias, spec.k, spec.s, score=spec.score)
    need = sorted(set(int(e) for t in sample for e in idx[t]))
    experts = {e: host_expert(spec, e) for e in need}
    shared = host_expert(spec, spec.E) if spec.f_shared else None
    return oracle.layer(spec.E, spec.k, spec.d, spec.f, spec.f_shared, spec.fmt, spec.s,
                        experts, shared, x, logits, bias, want=sample, score=spec.score)


CASES = [
    ("fused_t1", _spec(), 1, 0),
    ("fused_t2", _spec(), 2, 0),
    ("gemv_t9", _spec(), 9, 0),
    ("tc_t40", _spec(E=16, k=4, d=512, f=256, f_shared=256), 40, "tc"),
    ("q2_t13", _spec(E=48, k=8, d=1024, f=256, f_shared=256, fmt=1, s=1.0), 13, 0),
    ("fp4_tc_t40", _spec(E=16, k=4, d=512, f=256, f_shared=256, fmt=2, s=1.0), 40, "tc"),
    ("decode_shape_t1", synth.GLM_LAYER_E32, 1, 0),
    ("decode_shape_t16", synth.GLM_LAYER_E32, 16, 0),
]


@pytest.mark.parametrize("name,spec,T,fl", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("world", [2, 3])
def test_rank_partials_sum_to_the_layer(gpu, name, spec, T, fl, world):
    layer = device_layer(spec, gpu)
    flags = moe.FLAG_FORCE_TC if fl == "tc" else 0
    desc = layer.desc(flags)
    logits, x = synth.token_inputs(spec, 70 + T, T)
    bias = synth.bias(spec)
    x_d, l_d, b_d = (torch.from_numpy(a).to(gpu) for a in (x, logits, bias))
    ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=gpu)
    y_full = torch.empty((T, spec.d), dtype=torch.float32, device=gpu)
    moe.layer(desc, layer.weights, x_d, l_d, b_d, y_full, ws)
    y_sum = torch.zeros_like(y_full)
    for r, (lo, hi) in enumerate(expert_ranges(spec.E, world)):
        w_r, keep = _owned_weights(layer, lo, hi, gpu)
        y_r = torch.full_like(y_full, float("nan"))
        moe.layer_experts(desc, w_r, x_d, l_d, b_d, y_r, ws, lo, hi, r == 0)
        torch.cuda.synchronize()
        assert moe.check_device_error(ws) == 0, (r, lo, hi)
        assert torch.isfinite(y_r).all()
        y_sum += y_r
        del keep
    torch.cuda.synchronize()
    sample = list(range(T)) if T <= 16 else [0, T // 2, T - 1]
    ref = _oracle_y(spec, x, logits, bias, sample)
    g, f = y_sum.cpu().numpy(), y_full.cpu().numpy()
    for t in sample:
        assert np.abs(g[t] - ref.y[t]).max() / np.abs(ref.y[t]).max() <= Y_TOL, t
    # moe_layer's y within the same tolerance (a rank's share of the experts can
    # fall under the tensor-core dispatch rule where the whole layer does not,
    # and the two paths' fp32 orders can move an h code by one step)
    assert (np.abs(g - f).max(axis=1) / np.abs(f).max(axis=1)).max() <= Y_TOL


def test_unowned_expert_without_a_slot_is_never_read(gpu):
    """With every unowned expert mapped out of range, an owned-range call runs
    clean (the unowned slots are not read), while a full-range call on the same
    weights flags the bad slot."""
    spec = _spec()
    layer = device_layer(spec, gpu)
    desc = layer.desc()
    T = 6
    logits, x = synth.token_inputs(spec, 5, T)
    x_d, l_d = torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu)
    b_d = torch.from_numpy(synth.bias(spec)).to(gpu)
    ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=gpu)
    lo, hi = 0, spec.E // 2
    w_r, keep = _owned_weights(layer, lo, hi, gpu)
    y = torch.empty((T, spec.d), dtype=torch.float32, device=gpu)
    moe.layer_experts(desc, w_r, x_d, l_d, b_d, y, ws, lo, hi, True)
    assert moe.check_device_error(ws) == 0
    moe.layer(desc, w_r, x_d, l_d, b_d, y, ws)
    assert moe.check_device_error(ws) == 6  # MOE_ERR_DEVICE_CHECK
    del keep


def test_empty_range_is_the_shared_expert(gpu):
    spec = _spec()
    layer = device_layer(spec, gpu)
    desc = layer.desc()
    for T in (1, 7):
        logits, x = synth.token_inputs(spec, 9, T)
        x_d, l_d = torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu)
        b_d = torch.from_numpy(synth.bias(spec)).to(gpu)
        ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=gpu)
        y = torch.empty((T, spec.d), dtype=torch.float32, device=gpu)
        moe.layer_experts(desc, layer.weights, x_d, l_d, b_d, y, ws, 3, 3, True)
        torch.cuda.synchronize()
        sh = host_expert(spec, spec.E)
        for t in range(T):
            xq, xs = oracle.quantize(x[t])
            o = oracle.expert_row(oracle.FMT_Q8_0, spec.d, spec.f_shared, sh, xq, xs)[2]
            g = y[t].cpu().numpy()
            assert np.abs(g - o).max() / np.abs(o).max() <= Y_TOL
        with pytest.raises(moe.MoeError):
            moe.layer_experts(desc, layer.weights, x_d, l_d, b_d, y, ws, 5, 3, True)


@pytest.mark.parametrize("T", [1, 24])
def test_prefill_schedule_on_one_gpu(gpu, T):
    """The prefill schedule's GPU bindings (moe_route for the dispatch plan,
    moe_layer_experts for the owners and the shared expert) at world size 1:
    the exchanges are copies, the result is the layer."""
    spec = _spec()
    layer = device_layer(spec, gpu)
    b_d = torch.from_numpy(synth.bias(spec)).to(gpu)
    ep = ExpertParallel.for_layer(layer, b_d, 0, 1)
    logits, x = synth.token_inputs(spec, 12, T)
    x_d, l_d = torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu)
    y_p = ep.prefill(x_d, l_d)
    y_d = ep.decode(x_d, l_d)
    y = layer.forward(x_d, l_d, b_d).y
    torch.cuda.synchronize()
    f = y.cpu().numpy()
    for g in (y_p.cpu().numpy(), y_d.cpu().numpy()):
        assert (np.abs(g - f).max(axis=1) / np.abs(f).max(axis=1)).max() <= 1e-5
