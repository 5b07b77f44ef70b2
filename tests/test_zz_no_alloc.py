"""moe_layer_noalloc: the layer for callers that cannot allocate device memory
(an engine that reserved its whole device arena up front, plugins and plain-C
hosts without an allocator, paths that must not touch the allocator).  Its
scratch is the library's fixed 16 MiB device array, so these checks call it
through the C ABI, compare it bit for bit with moe_layer on a caller
workspace, and read its device error word with moe_check_device_error(NULL).

This file is collected last on purpose (its name sorts last)."""
import numpy as np
import pytest
import torch

import synth
from parity import Y_TOL

pytestmark = pytest.mark.gpu


def _layer(spec, dev):
    from routed_expert_decode_gb300 import moe

    t = synth.fill_layer_device(spec, dev)
    return moe.Layer(spec.E, spec.k, spec.d, spec.f, spec.f_shared, spec.fmt, spec.s, t, dev)


@pytest.mark.parametrize("spec,T", [
    (synth.LayerSpec("na_small", E=64, k=4, d=512, f=256, f_shared=256, fmt=0, s=2.5,
                     zipf_beta=0.4), 9),
    (synth.GLM_LAYER_E32, 1),
    (synth.GLM_LAYER_E32, 16),
    (synth.LayerSpec("na_q2", E=48, k=8, d=1024, f=384, f_shared=256, fmt=1, s=1.0,
                     zipf_beta=0.4), 5),
    (synth.LayerSpec("na_fp4", E=16, k=4, d=512, f=256, f_shared=256, fmt=2, s=1.0,
                     zipf_beta=0.4), 40),
], ids=["e64_t9", "decode_shape_t1", "decode_shape_t16", "q2_t5", "fp4_t40"])
def test_noalloc_matches_workspace_entry_twice(gpu, spec, T):
    """Same kernels, same inputs: the output equals moe_layer's bit for bit, on
    two calls in a row, and the static scratch's error word stays clear."""
    from routed_expert_decode_gb300 import moe

    layer = _layer(spec, gpu)
    desc = layer.desc()
    bias = torch.from_numpy(synth.bias(spec)).to(gpu)
    for seed in (21, 22):  # two calls in a row, different tokens
        logits, x = synth.token_inputs(spec, seed, T)
        x_d, l_d = torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu)
        ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=gpu)
        y_ref = torch.empty((T, spec.d), dtype=torch.float32, device=gpu)
        moe.layer(desc, layer.weights, x_d, l_d, bias, y_ref, ws)
        y = torch.full((T, spec.d), float("nan"), dtype=torch.float32, device=gpu)
        moe.layer_noalloc(desc, layer.weights, x_d, l_d, bias, y)
        assert moe.check_device_error(None) == 0
        torch.cuda.synchronize()
        a, b = y.cpu().numpy(), y_ref.cpu().numpy()
        assert np.isfinite(a).all()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        err = np.abs(a - b).max(axis=1) / np.abs(b).max(axis=1)
        assert err.max() <= Y_TOL, err.max()


def test_noalloc_reports_device_errors_and_recovers(gpu):
    """A caller with no workspace can still read the device error word: a
    stalled fused call (the failure-detection switch: its bounded waits run
    out, nothing faults) reports MOE_ERR_TIMEOUT through
    check_device_error(None), which also zeroes the scratch's counters, so the
    next call on the same static scratch is correct again."""
    from routed_expert_decode_gb300 import moe

    spec = synth.LayerSpec("na_stall", E=64, k=4, d=512, f=256, f_shared=256, fmt=0, s=2.5,
                           zipf_beta=0.4)
    layer = _layer(spec, gpu)
    logits, x = synth.token_inputs(spec, 5, 1)
    x_d, l_d = torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu)
    bias = torch.from_numpy(synth.bias(spec)).to(gpu)
    stall = layer.desc(moe.FLAG_TEST_STALL)
    assert moe.layer_path(stall, 1) == "fused_decode"
    y = torch.empty((1, spec.d), dtype=torch.float32, device=gpu)
    moe.layer_noalloc(stall, layer.weights, x_d, l_d, bias, y)
    assert moe.check_device_error(None) == 5  # MOE_ERR_TIMEOUT
    ws = torch.zeros(moe.workspace_size(layer.desc(), 1), dtype=torch.uint8, device=gpu)
    y_ref = torch.empty_like(y)
    moe.layer(layer.desc(), layer.weights, x_d, l_d, bias, y_ref, ws)
    for _ in range(2):
        moe.layer_noalloc(layer.desc(), layer.weights, x_d, l_d, bias, y)
        assert moe.check_device_error(None) == 0
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)


def test_noalloc_rejects_oversized_batches(gpu):
    from routed_expert_decode_gb300 import moe

    spec = synth.GLM_LAYER_E32
    layer = _layer(spec, gpu)
    desc = layer.desc()
    T = 512
    assert moe.workspace_size(desc, T) > moe.NOALLOC_SCRATCH_BYTES
    logits, x = synth.token_inputs(spec, 1, T)
    x_d, l_d = torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu)
    y = torch.zeros((T, spec.d), dtype=torch.float32, device=gpu)
    with pytest.raises(moe.MoeError) as ei:
        moe.layer_noalloc(desc, layer.weights, x_d, l_d,
                          torch.from_numpy(synth.bias(spec)).to(gpu), y)
    assert ei.value.status == 3
    assert "16 MiB" in moe.lib().moe_last_error().decode()
    torch.cuda.synchronize()
    assert (y == 0).all()
