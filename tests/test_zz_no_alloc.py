"""moe_layer_noalloc: the layer for callers that cannot allocate device memory
(an engine that reserved its whole device arena up front, plugins and plain-C
hosts without an allocator, paths that must not touch the allocator).  Its
scratch is the library's fixed 16 MiB device array, so these checks call it
through the C ABI and compare it with moe_layer on a caller workspace.

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
], ids=["e64_t9", "decode_shape_t1", "decode_shape_t16", "q2_t5"])
def test_noalloc_matches_workspace_entry_twice(gpu, spec, T):
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
        torch.cuda.synchronize()
        a, b = y.cpu().numpy(), y_ref.cpu().numpy()
        assert np.isfinite(a).all()
        err = np.abs(a - b).max(axis=1) / np.abs(b).max(axis=1)
        assert err.max() <= Y_TOL, err.max()


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
