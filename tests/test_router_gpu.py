"""Router front end on the GPU (pytest -m gpu): the router logits GEMM in the
library's fixed fp32 order must lie within that order's fp32 error bound of the
oracle's logit (the exact dot rounded once), both GPU implementations of the
order (moe_router_logits, and the router inside the fused decode kernel of
moe_layer_from_x) must give the same bits, and the DeepSeek scoring
sqrt(softplus(l)) (top-6, scale 1.5, E = 384: "256 experts, 512 lines",
section "The constant that always said 256") must pick the oracle's experts on
both the fused decode path and the multi-kernel path -- on the direct-logits
path unconditionally, on the from-x paths given the GPU's own logits."""
import numpy as np
import pytest
import torch

import synth
from parity import check_router_logits, device_layer, run_case
from routed_expert_decode_gb300 import moe

pytestmark = pytest.mark.gpu


def _spec(**kw):
    base = dict(name="r", E=64, k=8, d=512, f=256, f_shared=256, fmt=0, s=2.5, zipf_beta=0.0)
    base.update(kw)
    return synth.LayerSpec(**base)


@pytest.mark.parametrize("T,E,d", [(1, 256, 6144), (5, 384, 1024), (3, 37, 96), (64, 192, 4096)])
def test_router_logits_within_fp32_bound(gpu, T, E, d):
    rng = np.random.default_rng(T + E + d)
    x = rng.normal(size=(T, d)).astype(np.float32)
    w_r = (rng.normal(size=(E, d)) / np.sqrt(d)).astype(np.float32)
    out = torch.full((T, E), float("nan"), dtype=torch.float32, device=gpu)
    desc = moe.make_desc(E, min(8, E), d, 256, 0, 0, 1.0)
    moe.router_logits(desc, torch.from_numpy(w_r).to(gpu), torch.from_numpy(x).to(gpu), out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = check_router_logits(x, w_r, got)
    print("router logits equal to the rounded exact dot:", float((got == ref).mean()))


def test_router_logits_cancellation_within_bound(gpu):
    """Terms that cancel: the kernel's fp32 order may lose the small term (it
    adds the segment totals 2^24, 1, -2^24 in order), the oracle keeps it; the
    difference stays inside the order's error bound."""
    d = 3072
    x = np.zeros((1, d), np.float32)
    w = np.zeros((1, d), np.float32)
    x[0, [0, 1024, 2048]] = 1.0
    w[0, 0], w[0, 1024], w[0, 2048] = 2.0 ** 24, 1.0, -(2.0 ** 24)
    out = torch.full((1, 1), float("nan"), dtype=torch.float32, device=gpu)
    desc = moe.make_desc(1, 1, d, 256, 0, 0, 1.0)
    moe.router_logits(desc, torch.from_numpy(w).to(gpu), torch.from_numpy(x).to(gpu), out)
    torch.cuda.synchronize()
    check_router_logits(x, w, out.cpu().numpy())


@pytest.mark.parametrize("spec,T", [(synth.GLM_LAYER_E32, 1), (synth.GLM_LAYER_E32, 2)],
                         ids=["t1", "t2"])
def test_router_implementations_agree_bit_for_bit(gpu, spec, T):
    """The logits the fused decode kernel computes inside moe_layer_from_x equal
    moe_router_logits' bit for bit: both follow the library's one fp32 order."""
    layer = device_layer(spec, gpu)
    w_r = torch.from_numpy(synth.router_weights(spec)).to(gpu)
    bias = torch.from_numpy(synth.bias(spec)).to(gpu)
    for seed in (1, 2, 3):
        _, x = synth.token_inputs(spec, seed, T)
        x_d = torch.from_numpy(x).to(gpu)
        l_sep = torch.full((T, spec.E), float("nan"), dtype=torch.float32, device=gpu)
        l_fused = torch.full_like(l_sep, float("nan"))
        moe.router_logits(layer.desc(), w_r, x_d, l_sep)
        layer.forward_from_x(x_d, w_r, bias, l_fused)
        torch.cuda.synchronize()
        assert torch.equal(l_sep.view(torch.int32), l_fused.view(torch.int32)), seed


def test_router_logits_rejects_bad_args(gpu):
    desc = moe.make_desc(16, 4, 64, 64, 0, 0, 1.0)
    x = torch.zeros((2, 64), dtype=torch.float32, device=gpu)
    w = torch.zeros((16, 64), dtype=torch.float32, device=gpu)
    out = torch.zeros((2, 16), dtype=torch.float32, device=gpu)
    bad = moe.make_desc(16, 4, 64, 64, 0, 0, 1.0, score=7)
    with pytest.raises(moe.MoeError):
        moe.router_logits(bad, w, x, out)
    moe.router_logits(desc, w, x, out)  # well-formed call works
    torch.cuda.synchronize()


DS_SMALL = _spec(name="ds_small", E=384, k=6, d=1024, f=256, f_shared=256, s=1.5, score=1)


@pytest.mark.parametrize("T", [1, 2, 9])
def test_deepseek_scoring_layer(gpu, T):
    """sqrt(softplus) routing with E=384, k=6, s=1.5: T <= 2 on the fused kernel,
    T = 9 on the multi-kernel path; bit-exact picks, y within tolerance."""
    layer = device_layer(DS_SMALL, gpu)
    assert moe.layer_path(layer.desc(), T) == ("fused_decode" if T <= 2 else "multi_kernel")
    for seed in (1, 2):
        print("ds", T, seed, run_case(DS_SMALL, T, seed=seed, device=gpu))


@pytest.mark.parametrize("spec,T", [(_spec(name="glm_router"), 1), (_spec(name="glm_router"), 6),
                                    (DS_SMALL, 1)], ids=["sigmoid_t1", "sigmoid_t6", "ds_t1"])
def test_router_front_end_layer(gpu, spec, T):
    """x -> router GEMM -> scoring -> layer: logits within the fp32 bound, then
    full parity on the GPU's logits."""
    print("router", spec.name, T, run_case(spec, T, seed=4, device=gpu, router=True))


@pytest.mark.parametrize("router", [True, "fused"], ids=["separate", "fused"])
def test_deepseek_full_size_decode(gpu, router):
    """The full DeepSeek-style layer (E=384, k=6, d=6144, f=2048, shared 2048) at
    T=1 through the router GEMM, on the fused kernel."""
    print("ds_full", run_case(synth.DS_LAYER, 1, seed=0, device=gpu, router=router))


@pytest.mark.parametrize("spec,T", [(_spec(name="glm_router"), 1), (_spec(name="glm_router"), 2),
                                    (_spec(name="glm_router"), 6), (DS_SMALL, 1), (DS_SMALL, 2),
                                    (_spec(name="odd_router", E=37, k=5, d=768, f=512), 2)],
                         ids=["sigmoid_t1", "sigmoid_t2", "sigmoid_t6", "ds_t1", "ds_t2",
                              "e37_t2"])
def test_layer_from_x(gpu, spec, T):
    """moe_layer_from_x: logits within the fp32 bound of the oracle's router
    GEMM, then full parity of the layer on the GPU's logits (fused kernel at
    T <= 2, taps on)."""
    layer = device_layer(spec, gpu)
    assert moe.layer_path(layer.desc(), T) == ("fused_decode" if T <= 2 else "multi_kernel")
    for seed in (4, 5):
        print("from_x", spec.name, T, run_case(spec, T, seed=seed, device=gpu, router="fused"))


def test_layer_from_x_repeated_calls(gpu):
    """The fused kernel's router arrival counter is left zeroed by every call:
    back-to-back calls on one workspace give identical logits and y."""
    spec = _spec(name="glm_router")
    layer = device_layer(spec, gpu)
    w_r = torch.from_numpy(synth.router_weights(spec)).to(gpu)
    bias = torch.from_numpy(synth.bias(spec)).to(gpu)
    outs = []
    for _ in range(3):
        _, x = synth.token_inputs(spec, 7, 1)
        l_dev = torch.empty((1, spec.E), dtype=torch.float32, device=gpu)
        out = layer.forward_from_x(torch.from_numpy(x).to(gpu), w_r, bias, l_dev)
        torch.cuda.synchronize()
        outs.append((l_dev.cpu().numpy().copy(), out.y.cpu().numpy().copy()))
    assert moe.check_device_error(layer.workspace(1, 0)) == 0
    for l_, y_ in outs[1:]:
        assert np.array_equal(l_.view(np.uint32), outs[0][0].view(np.uint32))
        assert np.array_equal(y_.view(np.uint32), outs[0][1].view(np.uint32))


def test_layer_from_x_rejects_bad_args(gpu):
    spec = _spec(name="glm_router")
    layer = device_layer(spec, gpu)
    x = torch.zeros((1, spec.d), dtype=torch.float32, device=gpu)
    bias = torch.zeros((spec.E,), dtype=torch.float32, device=gpu)
    l_dev = torch.zeros((1, spec.E), dtype=torch.float32, device=gpu)
    ws = layer.workspace(1, 0)
    y = torch.zeros((1, spec.d), dtype=torch.float32, device=gpu)
    with pytest.raises(moe.MoeError):
        moe.layer_from_x(layer.desc(), layer.weights, None, x, bias, l_dev, y, ws)
    w_r = torch.zeros((spec.E, spec.d), dtype=torch.float32, device=gpu)
    moe.layer_from_x(layer.desc(), layer.weights, w_r, x, bias, l_dev, y, ws)
    torch.cuda.synchronize()
