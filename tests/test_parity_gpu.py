"""CUDA path vs the CPU oracle, through the C ABI, on a GB300 (sm_103a)."""
import numpy as np
import pytest
import torch

import synth
from parity import Y_TOL, run_case, device_layer, poison_workspace

pytestmark = pytest.mark.gpu


def _spec(**kw):
    base = dict(name="t", E=16, k=4, d=256, f=128, f_shared=0, fmt=0, s=1.0, zipf_beta=0.0)
    base.update(kw)
    return synth.LayerSpec(**base)


# ---------------------------------------------------------------- small layers, all tokens
SMALL = [
    ("tiny_t4", synth.TINY, 4),
    ("tiny_ragged_t37", synth.TINY, 37),
    ("shared_e64", _spec(E=64, k=4, d=512, f=256, f_shared=256, s=2.5, zipf_beta=0.4), 9),
    ("e192_q2", _spec(E=192, k=8, d=512, f=192, f_shared=160, fmt=1, zipf_beta=0.4), 13),
    ("e192_fp4", _spec(E=192, k=8, d=512, f=192, f_shared=160, fmt=2, zipf_beta=0.4), 13),
    ("e384_k6", _spec(E=384, k=6, d=256, f=96, f_shared=64, s=1.5), 7),
    ("e256_d6144", _spec(E=256, k=8, d=6144, f=64, f_shared=96, s=2.5, zipf_beta=0.4), 3),
    ("k1_s1", _spec(E=16, k=1, d=256, f=128), 6),
    ("k_eq_E", _spec(E=8, k=8, d=128, f=64, f_shared=32), 5),
    ("e1024_k32", _spec(E=1024, k=32, d=128, f=32, f_shared=0), 3),
    ("many_rows_per_expert", _spec(E=4, k=2, d=256, f=128, f_shared=64), 40),
    # d not a multiple of 128: gate/up on the register-streaming GEMV (down
    # streamed where its rows copy in whole 16-byte units: Q8_0 and e2m1 here,
    # the 2-bit layer's 24-byte rows on the register GEMV)
    ("d224_gemv_gateup", _spec(E=16, k=4, d=224, f=96, f_shared=64, s=2.5), 7),
    ("q2_d224_gemv_gateup", _spec(E=24, k=4, d=224, f=96, f_shared=64, fmt=1, s=1.0), 9),
    ("fp4_d160_gemv_gateup", _spec(E=24, k=4, d=160, f=128, f_shared=64, fmt=2, s=1.0), 9),
]


@pytest.mark.parametrize("name,spec,T", SMALL, ids=[s[0] for s in SMALL])
def test_small_layers(gpu, name, spec, T):
    rep = run_case(spec, T, seed=11, device=gpu)
    print(name, rep)


def test_tie_logits_pick_lower_index(gpu):
    """Equal logits and bias: every token must take experts 0..k-1 in order."""
    from routed_expert_decode_gb300 import moe

    spec = _spec(E=32, k=4)
    layer = device_layer(spec, gpu)
    T = 3
    logits = torch.zeros((T, 32), dtype=torch.float32, device=gpu)
    bias = torch.zeros(32, dtype=torch.float32, device=gpu)
    x = torch.ones((T, spec.d), dtype=torch.float32, device=gpu)
    out = layer.forward(x, logits, bias)
    torch.cuda.synchronize()
    assert out.idx.cpu().tolist() == [[0, 1, 2, 3]] * T
    assert np.allclose(out.w.cpu().numpy(), 0.25)


@pytest.mark.parametrize("E,k,T", [(32, 4, 1), (300, 8, 2), (600, 4, 2)])
def test_fused_selection_ties_and_infinite_bias(gpu, E, k, T):
    """The fused decode kernel's top-k (register keys for E <= 512, a shared
    memory scan above): equal scores go to the lower expert, and with all but two
    biases at -inf the two finite experts come first, then the lowest-indexed
    -inf ones -- the oracle's order in both cases."""
    import oracle
    from routed_expert_decode_gb300 import moe

    spec = _spec(E=E, k=k, d=256, f=256)
    layer = device_layer(spec, gpu)
    assert moe.layer_path(layer.desc(), T) == "fused_decode"
    rng = np.random.default_rng(E)
    x = torch.from_numpy(rng.normal(size=(T, spec.d)).astype(np.float32)).to(gpu)
    logits = np.zeros((T, E), dtype=np.float32)
    bias = np.zeros(E, dtype=np.float32)
    out = layer.forward(x, torch.from_numpy(logits).to(gpu), torch.from_numpy(bias).to(gpu))
    torch.cuda.synchronize()
    assert out.idx.cpu().tolist() == [list(range(k))] * T
    bias[:] = -np.inf
    bias[[E // 2, E - 1]] = 0.0
    logits = rng.normal(size=(T, E)).astype(np.float32)
    out = layer.forward(x, torch.from_numpy(logits).to(gpu), torch.from_numpy(bias).to(gpu))
    torch.cuda.synchronize()
    ref_idx, ref_w = oracle.route(logits, bias, k, spec.s)
    assert np.array_equal(out.idx.cpu().numpy(), ref_idx)
    assert np.allclose(out.w.cpu().numpy(), ref_w, rtol=4e-6, atol=0)
    assert moe.check_device_error(layer.workspace(T, 0)) == 0


def test_zero_tokens(gpu):
    spec = synth.TINY
    layer = device_layer(spec, gpu)
    x = torch.empty((0, spec.d), dtype=torch.float32, device=gpu)
    lg = torch.empty((0, spec.E), dtype=torch.float32, device=gpu)
    out = layer.forward(x, lg, torch.zeros(spec.E, device=gpu))
    torch.cuda.synchronize()
    assert out.y.shape == (0, spec.d)
    assert out.off.cpu().tolist() == [0] * (spec.E + 1)


def test_zero_activation_block(gpu):
    """An all-zero 32-block quantises to scale 0 and codes 0 (no division by zero)."""
    spec = synth.TINY
    layer = device_layer(spec, gpu)
    logits, x = synth.token_inputs(spec, 3, 2)
    x[:, 32:96] = 0.0
    out = layer.forward(torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu),
                        torch.from_numpy(synth.bias(spec)).to(gpu))
    torch.cuda.synchronize()
    assert (out.xs.cpu().numpy()[:, 1:3] == 0).all()
    assert (out.xq.cpu().numpy()[:, 32:96] == 0).all()
    assert np.isfinite(out.y.cpu().numpy()).all()


def test_deterministic_across_runs(gpu):
    spec = _spec(E=64, k=4, d=512, f=256, f_shared=256, s=2.5, zipf_beta=0.4)
    layer = device_layer(spec, gpu)
    logits, x = synth.token_inputs(spec, 5, 21)
    args = [torch.from_numpy(a).to(gpu) for a in (x, logits, synth.bias(spec))]
    y1 = layer.forward(*args).y.clone()
    y2 = layer.forward(*args).y.clone()
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("T,fl", [(1, 0), (1, "gemv"), (7, 0), (40, "tc")])
def test_x_and_y_only_float_aligned(gpu, T, fl):
    """x and y at an odd float offset (4-byte, not 16-byte aligned): the fused
    kernel, which reads x in 16-byte vectors, is not used and the multi-kernel
    kernels read x and write y element by element there; the outputs equal the
    aligned multi-kernel call's bit for bit."""
    from routed_expert_decode_gb300 import moe

    spec = _spec(E=32, k=4, d=512, f=256, f_shared=256, s=2.5, zipf_beta=0.4)
    layer = device_layer(spec, gpu)
    flags = {0: 0, "gemv": moe.FLAG_FORCE_GEMV, "tc": moe.FLAG_FORCE_TC}[fl]
    logits, x = synth.token_inputs(spec, 31, T)
    l_d = torch.from_numpy(logits).to(gpu)
    b_d = torch.from_numpy(synth.bias(spec)).to(gpu)
    n = T * spec.d
    xbuf = torch.zeros(n + 4, dtype=torch.float32, device=gpu)
    xbuf[1:1 + n] = torch.from_numpy(x).to(gpu).reshape(-1)
    x_odd = xbuf[1:1 + n].view(T, spec.d)
    x_al = torch.from_numpy(x).to(gpu)
    ybuf = torch.full((n + 4,), float("nan"), dtype=torch.float32, device=gpu)
    y_odd = ybuf[1:1 + n].view(T, spec.d)
    y_al = torch.empty((T, spec.d), dtype=torch.float32, device=gpu)
    # the aligned reference on the multi-kernel path (the unaligned call's path)
    ref_desc = layer.desc(flags if flags else moe.FLAG_FORCE_GEMV)
    desc = layer.desc(flags)
    nws = max(moe.workspace_size(desc, T), moe.workspace_size(ref_desc, T))
    ws = torch.zeros(nws, dtype=torch.uint8, device=gpu)
    moe.layer(ref_desc, layer.weights, x_al, l_d, b_d, y_al, ws)
    moe.layer(desc, layer.weights, x_odd, l_d, b_d, y_odd, ws)
    torch.cuda.synchronize()
    assert moe.check_device_error(ws) == 0
    assert x_odd.data_ptr() % 16 != 0 and y_odd.data_ptr() % 16 != 0
    assert torch.equal(y_odd, y_al)
    assert torch.isnan(ybuf[0]) and torch.isnan(ybuf[1 + n])  # nothing written outside y


@pytest.mark.parametrize("T,fl", [(7, 0), (40, "tc")])
def test_two_bit_planes_only_8_byte_aligned(gpu, T, fl):
    """2-bit routed code planes at an 8-byte (not 16-byte) offset, as moe_weights
    allows them: the paths that need 16-byte aligned planes (the streamed GEMV's
    bulk copies, the tensor maps) are not taken.  The block-dot taps equal the
    aligned layer's bit for bit and y agrees within the layer tolerance."""
    from routed_expert_decode_gb300 import moe

    spec = _spec(E=32, k=4, d=512, f=256, f_shared=256, fmt=1, s=1.0, zipf_beta=0.4)
    layer = device_layer(spec, gpu)
    keep = {}
    w = moe.MoeWeights()
    for name in ("gate", "up", "down"):
        q = layer.tensors[name + "_q"].reshape(-1).view(torch.uint8)
        buf = torch.zeros(q.numel() + 16, dtype=torch.uint8, device=gpu)
        buf[8:8 + q.numel()] = q
        keep[name] = buf
        setattr(w, name, moe.MoeMat(buf.data_ptr() + 8, layer.tensors[name + "_s"].data_ptr()))
    for name in ("s_gate", "s_up", "s_down"):
        setattr(w, name, getattr(layer.weights, name))
    w.expert_slot = layer.weights.expert_slot
    w.n_slots = layer.weights.n_slots
    assert w.gate.q % 16 == 8
    flags = moe.FLAG_DEBUG_TAPS | (moe.FLAG_FORCE_TC if fl == "tc" else 0)
    ref_flags = moe.FLAG_DEBUG_TAPS | moe.FLAG_FORCE_GEMV
    logits, x = synth.token_inputs(spec, 17, T)
    x_d, l_d = torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu)
    b_d = torch.from_numpy(synth.bias(spec)).to(gpu)
    out = {}
    for key, fls, wts in (("ref", ref_flags, layer.weights), ("odd", flags, w)):
        desc = layer.desc(fls)
        ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=gpu)
        y = torch.empty((T, spec.d), dtype=torch.float32, device=gpu)
        moe.layer(desc, wts, x_d, l_d, b_d, y, ws)
        torch.cuda.synchronize()
        assert moe.check_device_error(ws) == 0, key
        L = moe.workspace_layout(desc, T)
        slots = T * spec.k + T
        n_gu = slots * 2 * L.n_tap * (spec.d // 32) * 4
        n_dn = slots * L.n_tap * (max(spec.f, spec.f_shared) // 32) * 4
        out[key] = (y.cpu().numpy(), ws[L.tap_gu:L.tap_gu + n_gu].cpu(),
                    ws[L.tap_dn:L.tap_dn + n_dn].cpu())
    assert torch.equal(out["ref"][1], out["odd"][1])
    assert torch.equal(out["ref"][2], out["odd"][2])
    g, f = out["odd"][0], out["ref"][0]
    assert (np.abs(g - f).max(axis=1) / np.abs(f).max(axis=1)).max() <= Y_TOL
    del keep


@pytest.mark.parametrize("T,fl", [(1, 0), (7, 0), (40, "tc")])
def test_q8_scale_planes_only_2_byte_aligned(gpu, T, fl):
    """Q8_0 scale planes (routed and shared) at a 2-byte offset, as moe_weights
    allows them: the fused decode kernel, the streamed GEMV and the tensor maps,
    which copy scales in 16-byte units, are not used.  The block-dot taps equal
    the aligned layer's bit for bit and y agrees within the layer tolerance."""
    from routed_expert_decode_gb300 import moe

    spec = _spec(E=32, k=4, d=512, f=256, f_shared=256, s=2.5, zipf_beta=0.4)
    layer = device_layer(spec, gpu)
    keep = {}
    w = moe.MoeWeights()
    for name, key in (("gate", "gate"), ("up", "up"), ("down", "down"),
                      ("s_gate", "s_gate"), ("s_up", "s_up"), ("s_down", "s_down")):
        m = getattr(layer.weights, name)
        if name.startswith("s_"):
            sc = layer.tensors[key + "_s"] if key + "_s" in layer.tensors else None
        else:
            sc = layer.tensors[key + "_s"]
        if sc is None:
            setattr(w, name, m)
            continue
        flat = sc.reshape(-1).view(torch.uint8)
        buf = torch.zeros(flat.numel() + 32, dtype=torch.uint8, device=gpu)
        buf[2:2 + flat.numel()] = flat
        keep[name] = buf
        setattr(w, name, moe.MoeMat(m.q, buf.data_ptr() + 2))
    w.expert_slot = layer.weights.expert_slot
    w.n_slots = layer.weights.n_slots
    assert w.gate.scale % 16 == 2 and w.down.scale % 16 == 2
    flags = moe.FLAG_DEBUG_TAPS | (moe.FLAG_FORCE_TC if fl == "tc" else 0)
    ref_flags = moe.FLAG_DEBUG_TAPS | moe.FLAG_FORCE_GEMV
    logits, x = synth.token_inputs(spec, 19, T)
    x_d, l_d = torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu)
    b_d = torch.from_numpy(synth.bias(spec)).to(gpu)
    out = {}
    for key, fls, wts in (("ref", ref_flags, layer.weights), ("odd", flags, w)):
        desc = layer.desc(fls)
        ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=gpu)
        y = torch.empty((T, spec.d), dtype=torch.float32, device=gpu)
        moe.layer(desc, wts, x_d, l_d, b_d, y, ws)
        torch.cuda.synchronize()
        assert moe.check_device_error(ws) == 0, key
        L = moe.workspace_layout(desc, T)
        slots = T * spec.k + T
        n_gu = slots * 2 * L.n_tap * (spec.d // 32) * 4
        n_dn = slots * L.n_tap * (max(spec.f, spec.f_shared) // 32) * 4
        out[key] = (y.cpu().numpy(), ws[L.tap_gu:L.tap_gu + n_gu].cpu(),
                    ws[L.tap_dn:L.tap_dn + n_dn].cpu())
    assert torch.equal(out["ref"][1], out["odd"][1])
    assert torch.equal(out["ref"][2], out["odd"][2])
    g, f = out["odd"][0], out["ref"][0]
    assert (np.abs(g - f).max(axis=1) / np.abs(f).max(axis=1)).max() <= Y_TOL
    del keep


@pytest.mark.parametrize("T", [16, 40])
def test_streamed_gemv_repeatable_with_flushes(gpu, T):
    """The streamed GEMV's shared-memory ring (four stages read by three consumer
    groups in turn) under varying timing: 12 calls, each after an L2 flush,
    give the h codes and y of the first call bit for bit (every expert on the
    dp4a path: at T=40 FORCE_GEMV keeps the tensor cores off)."""
    from routed_expert_decode_gb300 import moe

    spec = synth.GLM_LAYER_E32
    layer = device_layer(spec, gpu)
    logits, x = synth.token_inputs(spec, 70 + T, T)
    args = [torch.from_numpy(a).to(gpu) for a in (x, logits, synth.bias(spec))]
    flush = torch.empty(2 * torch.cuda.get_device_properties(gpu).L2_cache_size,
                        dtype=torch.uint8, device=gpu)
    ref = layer.forward(*args, flags=moe.FLAG_FORCE_GEMV)
    y0, h0 = ref.y.clone(), ref.hq.clone()
    for i in range(12):
        flush.fill_(i)
        out = layer.forward(*args, flags=moe.FLAG_FORCE_GEMV)
        torch.cuda.synchronize()
        assert torch.equal(out.hq, h0) and torch.equal(out.y, y0), i


def test_ffn_entry_matches_layer(gpu):
    """moe_route + moe_ffn on caller buffers equals moe_layer."""
    from routed_expert_decode_gb300 import moe

    spec = _spec(E=64, k=4, d=512, f=256, f_shared=256, s=2.5, zipf_beta=0.4)
    layer = device_layer(spec, gpu)
    T = 10
    logits, x = synth.token_inputs(spec, 8, T)
    x_d, l_d = torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu)
    b_d = torch.from_numpy(synth.bias(spec)).to(gpu)
    ref = layer.forward(x_d, l_d, b_d).y.clone()
    idx = torch.empty((T, spec.k), dtype=torch.int32, device=gpu)
    w = torch.empty((T, spec.k), dtype=torch.float32, device=gpu)
    off = torch.empty(spec.E + 1, dtype=torch.int32, device=gpu)
    perm = torch.empty(T * spec.k, dtype=torch.int32, device=gpu)
    pos = torch.empty(T * spec.k, dtype=torch.int32, device=gpu)
    desc = layer.desc()
    moe.route(desc, l_d, b_d, idx, w, off, perm, pos)
    y = torch.empty((T, spec.d), dtype=torch.float32, device=gpu)
    ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=gpu)
    moe.ffn(desc, layer.weights, x_d, idx, w, off, perm, pos, y, ws)
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
    assert moe.check_device_error(ws) == 0


def test_ffn_rejects_inconsistent_routing_on_device(gpu):
    """Corrupted off/perm/idx are caught by the device-side check: the call
    reports MOE_ERR_DEVICE_CHECK, runs no expert and leaves y at zero."""
    from routed_expert_decode_gb300 import moe

    spec = _spec(E=16, k=4, d=256, f=128)
    layer = device_layer(spec, gpu)
    T = 4
    logits, x = synth.token_inputs(spec, 9, T)
    x_d, l_d = torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu)
    b_d = torch.from_numpy(synth.bias(spec)).to(gpu)
    idx = torch.empty((T, spec.k), dtype=torch.int32, device=gpu)
    w = torch.empty((T, spec.k), dtype=torch.float32, device=gpu)
    off = torch.empty(spec.E + 1, dtype=torch.int32, device=gpu)
    perm = torch.empty(T * spec.k, dtype=torch.int32, device=gpu)
    pos = torch.empty(T * spec.k, dtype=torch.int32, device=gpu)
    desc = layer.desc()
    moe.route(desc, l_d, b_d, idx, w, off, perm, pos)
    ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=gpu)
    y = torch.full((T, spec.d), 7.0, dtype=torch.float32, device=gpu)
    for corrupt in ("off", "perm", "idx"):
        o2, p2, i2 = off.clone(), perm.clone(), idx.clone()
        if corrupt == "off":
            o2[3] += 100
        elif corrupt == "perm":
            p2[0] = 10 ** 6
        else:
            i2[0, 0] = spec.E + 5
        moe.ffn(desc, layer.weights, x_d, i2, w, o2, p2, pos, y, ws)
        assert moe.check_device_error(ws) == 6, corrupt
        assert (y == 0).all()
    moe.ffn(desc, layer.weights, x_d, idx, w, off, perm, pos, y, ws)
    assert moe.check_device_error(ws) == 0


def test_device_fill_matches_host_generator(gpu):
    spec = synth.GLM_LAYER
    small = synth.LayerSpec("fillcheck", E=3, k=1, d=spec.d, f=256, f_shared=128, fmt=0, s=1.0,
                            zipf_beta=0.0)
    for sp in (small, synth.LayerSpec("fill2", E=2, k=1, d=512, f=96, f_shared=64, fmt=1, s=1.0,
                                      zipf_beta=0.0)):
        t = synth.fill_layer_device(sp, gpu)
        for e in range(sp.E):
            h = synth.expert_host(sp, e)
            for name in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
                dev = t[name][e].cpu().numpy()
                assert np.array_equal(dev.view(np.uint8), np.asarray(h[name]).view(np.uint8)), name
        hs = synth.expert_host(sp, sp.E)
        for name in ("gate_q", "gate_s", "down_q", "down_s"):
            dev = t["s_" + name].cpu().numpy()
            assert np.array_equal(dev.view(np.uint8), np.asarray(hs[name]).view(np.uint8))


# ---------------------------------------------------------------- full-size layers, sampled
def test_decode_t1_full_size(gpu):
    """The headline decode step on the fused kernel, with its block-dot taps:
    gate/up and down int32 block dots bit-exact against the oracle."""
    from routed_expert_decode_gb300 import moe

    layer = device_layer(synth.GLM_LAYER, gpu)
    assert moe.layer_path(layer.desc(moe.FLAG_DEBUG_TAPS), 1) == "fused_decode"
    for seed in (0, 1, 2):
        rep = run_case(synth.GLM_LAYER, 1, seed=seed, device=gpu)
        print("decode_t1", seed, rep)


def test_decode_t1_full_size_multi_kernel(gpu):
    """The same tokens through the multi-kernel (dp4a GEMV) path."""
    from routed_expert_decode_gb300 import moe

    for seed in (0, 1):
        rep = run_case(synth.GLM_LAYER, 1, seed=seed, device=gpu, flags=moe.FLAG_FORCE_GEMV)
        print("decode_t1 gemv", seed, rep)


def test_small_batch_t2_t16_full_size(gpu):
    print("batch_t2", run_case(synth.GLM_LAYER, 2, seed=0, device=gpu))
    print("batch_t16", run_case(synth.GLM_LAYER, 16, seed=0, device=gpu, sample=[0, 7, 15]))


def test_prefill_t512_full_size(gpu):
    print("prefill_t512", run_case(synth.GLM_LAYER, 512, seed=0, device=gpu,
                                   sample=[0, 255, 511]))


def test_q2_t64_full_size(gpu):
    """The 2-bit layer at T=64 (auto dispatch: the shared expert and the 2-bit
    experts with more than 6 rows on the tensor cores, when they fill the SMs)."""
    from routed_expert_decode_gb300 import moe

    layer = device_layer(synth.Q2_LAYER, gpu)
    assert moe.tc_min_rows(layer.desc(), 64) == 6
    print("q2_t64", run_case(synth.Q2_LAYER, 64, seed=0, device=gpu, sample=[0, 33, 63]))
    print("q2_t64 gemv", run_case(synth.Q2_LAYER, 64, seed=0, device=gpu, sample=[0, 63],
                                  flags=moe.FLAG_FORCE_GEMV))


def test_fp4_t64_full_size(gpu):
    """The e2m1 layer (the 2-bit layer's shape) at T=64, auto dispatch and
    dp4a-only: the same exact block dots on both paths (auto dispatch puts the
    experts with more than 4 rows on the tensor cores)."""
    from routed_expert_decode_gb300 import moe

    layer = device_layer(synth.E2M1_LAYER, gpu)
    assert moe.tc_min_rows(layer.desc(), 64) == 4
    print("fp4_t64", run_case(synth.E2M1_LAYER, 64, seed=0, device=gpu, sample=[0, 33, 63]))
    print("fp4_t64 gemv", run_case(synth.E2M1_LAYER, 64, seed=0, device=gpu, sample=[0, 63],
                                   flags=moe.FLAG_FORCE_GEMV))


# ---------------------------------------------------------------- fused decode kernel (T <= 2)
FUSED = [
    ("fused_e64_t1", _spec(E=64, k=4, d=512, f=256, f_shared=256, s=2.5, zipf_beta=0.4), 1),
    ("fused_e64_t2", _spec(E=64, k=4, d=512, f=256, f_shared=256, s=2.5, zipf_beta=0.4), 2),
    ("fused_noshared_t2", _spec(E=32, k=8, d=768, f=512, f_shared=0), 2),
    ("fused_wide_shared_t1", _spec(E=384, k=6, d=1024, f=256, f_shared=512, s=1.5), 1),
    ("fused_k32_t2", _spec(E=1024, k=32, d=1024, f=256, f_shared=256), 2),
]


@pytest.mark.parametrize("name,spec,T", FUSED, ids=[s[0] for s in FUSED])
def test_fused_small_layers(gpu, name, spec, T):
    from routed_expert_decode_gb300 import moe

    layer = device_layer(spec, gpu)
    assert moe.layer_path(layer.desc(), T) == "fused_decode"
    assert moe.layer_path(layer.desc(moe.FLAG_DEBUG_TAPS), T) == "fused_decode"
    for seed in (3, 4):
        rep = run_case(spec, T, seed=seed, device=gpu)
        print(name, seed, rep)


def test_fused_decode_full_size(gpu):
    from routed_expert_decode_gb300 import moe

    layer = device_layer(synth.GLM_LAYER, gpu)
    assert moe.layer_path(layer.desc(), 1) == "fused_decode"
    assert moe.layer_path(layer.desc(), 2) == "fused_decode"
    assert moe.layer_path(layer.desc(), 3) == "multi_kernel"
    assert moe.layer_path(layer.desc(moe.FLAG_DEBUG_TAPS), 2) == "fused_decode"
    for seed in (0, 1, 2, 3):
        print("fused t1", seed, run_case(synth.GLM_LAYER, 1, seed=seed, device=gpu))
    for seed in (0, 1):
        print("fused t2", seed, run_case(synth.GLM_LAYER, 2, seed=seed, device=gpu))


def test_decode_t1_every_bench_token(gpu):
    """Every token the decode benchmark times (its workload's token seeds), through
    the same untapped fused call: expert indices, routing weights, offsets,
    permutation and int8 activations against the oracle for each of them, and
    the whole bar (h codes within one step, y) on every tenth."""
    import oracle
    from parity import W_RTOL, compare_with_oracle
    from routed_expert_decode_gb300 import moe

    spec, T, seeds = synth.WORKLOADS["decode_t1"]
    assert T == 1 and len(seeds) == 100
    layer = device_layer(spec, gpu)
    assert moe.layer_path(layer.desc(), T) == "fused_decode"
    bias = synth.bias(spec)
    bias_d = torch.from_numpy(bias).to(gpu)
    worst = 0.0
    for i, seed in enumerate(seeds):
        logits, x = synth.token_inputs(spec, seed, T)
        out = layer.forward(torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu), bias_d)
        torch.cuda.synchronize()
        assert moe.check_device_error(layer.workspace(T, 0)) == 0
        g = {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in vars(out).items()}
        r_idx, r_w = oracle.route(logits, bias, spec.k, spec.s, score=spec.score)
        r_off, r_perm, r_pos = oracle.permute(r_idx, spec.E)
        r_xq, r_xs = oracle.quantize(x)
        assert np.array_equal(g["idx"].ravel(), r_idx.ravel()), f"seed {seed}: expert indices"
        assert np.allclose(g["w"].ravel(), r_w.ravel(), rtol=W_RTOL, atol=0), f"seed {seed}: weights"
        assert np.array_equal(g["off"].ravel(), r_off), f"seed {seed}: offsets"
        assert np.array_equal(g["perm"].ravel(), r_perm), f"seed {seed}: permutation"
        assert np.array_equal(g["pos"].ravel(), r_pos), f"seed {seed}: inverse permutation"
        assert np.array_equal(g["xq"].ravel(), r_xq), f"seed {seed}: int8 activations"
        assert np.array_equal(g["xs"].ravel(), r_xs), f"seed {seed}: activation scales"
        if i % 10 == 0:
            rep = compare_with_oracle(spec, T, x, logits, bias, g)
            worst = max(worst, rep["max_y_err"])
    print("decode_t1, 100 token seeds: worst sampled y error", worst)


def test_fused_matches_multi_kernel_and_repeats(gpu):
    """The fused kernel and the multi-kernel path agree (same routing, same
    int8 codes, y within fp32 summation order), the fused kernel is
    bit-identical from call to call, and its tapped variant (block dots stored
    on the side) gives the untapped kernel's y bit for bit."""
    from routed_expert_decode_gb300 import moe

    spec = synth.GLM_LAYER
    layer = device_layer(spec, gpu)
    bias = torch.from_numpy(synth.bias(spec)).to(gpu)
    for T in (1, 2):
        logits, x = synth.token_inputs(spec, 40 + T, T)
        args = [torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu), bias]
        a = layer.forward(*args)
        ya, ia, xa = a.y.clone(), a.idx.clone(), a.xq.clone()
        b = layer.forward(*args)
        assert torch.equal(b.y, ya)
        tp = layer.forward(*args, taps=True)
        assert torch.equal(tp.y, ya) and torch.equal(tp.hq, a.hq)
        m = layer.forward(*args, flags=moe.FLAG_FORCE_GEMV)
        torch.cuda.synchronize()
        assert torch.equal(m.idx, ia) and torch.equal(m.xq, xa)
        ym, yf = m.y.cpu().numpy(), ya.cpu().numpy()
        err = np.abs(ym - yf).max(axis=1) / np.abs(ym).max(axis=1)
        assert err.max() < 1e-4, err


def test_fused_wait_timeout_is_reported(gpu):
    """Failure detection without a GPU fault: with MOE_FLAG_TEST_STALL the router
    never publishes its result, every bounded wait runs out (~10 ms), the call
    reports MOE_ERR_TIMEOUT through the error word, and the next call works."""
    from routed_expert_decode_gb300 import moe

    spec = _spec(E=64, k=4, d=512, f=256, f_shared=256, s=2.5, zipf_beta=0.4)
    layer = device_layer(spec, gpu)
    logits, x = synth.token_inputs(spec, 5, 1)
    args = [torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu),
            torch.from_numpy(synth.bias(spec)).to(gpu)]
    desc = layer.desc(moe.FLAG_TEST_STALL)
    assert moe.layer_path(desc, 1) == "fused_decode"
    ws = torch.zeros(moe.workspace_size(desc, 1), dtype=torch.uint8, device=gpu)
    y = torch.empty((1, spec.d), dtype=torch.float32, device=gpu)
    moe.layer(desc, layer.weights, args[0], args[1], args[2], y, ws)
    assert moe.check_device_error(ws) == 5  # MOE_ERR_TIMEOUT
    moe.layer(layer.desc(), layer.weights, args[0], args[1], args[2], y, ws)
    assert moe.check_device_error(ws) == 0
    ref = layer.forward(*args, flags=moe.FLAG_FORCE_GEMV).y
    torch.cuda.synchronize()
    assert torch.allclose(y, ref, rtol=1e-4, atol=1e-6 * float(ref.abs().max()))


# ---------------------------------------------------------------- tensor-core expert path
TC_CASES = [
    ("tc_small_forced", _spec(E=16, k=4, d=256, f=256, f_shared=256, s=2.5, zipf_beta=0.4), 9),
    ("tc_ragged_rows", _spec(E=8, k=2, d=512, f=256, f_shared=256, s=1.0), 70),
    ("tc_d6144", _spec(E=16, k=4, d=6144, f=256, f_shared=256, s=2.5), 33),
    # 2-bit routed weights decoded to fp16 by the converters; the shared expert Q8_0
    ("tc_q2_forced", _spec(E=16, k=4, d=512, f=256, f_shared=256, fmt=1, s=1.0,
                           zipf_beta=0.4), 9),
    ("tc_q2_d4096", _spec(E=24, k=8, d=4096, f=512, f_shared=512, fmt=1, s=1.0), 33),
    ("tc_q2_noshared", _spec(E=8, k=2, d=1024, f=768, f_shared=0, fmt=1, s=1.0), 21),
    # e2m1 routed weights decoded to fp16 as twice their values (scale halved)
    ("tc_fp4_forced", _spec(E=16, k=4, d=512, f=256, f_shared=256, fmt=2, s=1.0,
                            zipf_beta=0.4), 9),
    ("tc_fp4_d4096", _spec(E=24, k=8, d=4096, f=512, f_shared=512, fmt=2, s=1.0), 33),
    ("tc_fp4_noshared", _spec(E=8, k=2, d=1024, f=768, f_shared=0, fmt=2, s=1.0), 21),
]


@pytest.mark.parametrize("name,spec,T", TC_CASES, ids=[c[0] for c in TC_CASES])
def test_tensor_core_path_forced(gpu, name, spec, T):
    """Every expert on tcgen05 (MOE_FLAG_FORCE_TC): int32 block dots read back
    from TMEM must equal the oracle's exactly; y within tolerance."""
    from routed_expert_decode_gb300 import moe

    rep = run_case(spec, T, seed=13, device=gpu, flags=moe.FLAG_FORCE_TC)
    print(name, rep)


def test_prefill_tensor_core_dispatch(gpu):
    """T=512 on the full layer: experts with more than 16 rows (and the shared
    expert) take the tensor-core path, the rest dp4a; sampled tokens vs the oracle."""
    from routed_expert_decode_gb300 import moe

    layer = device_layer(synth.GLM_LAYER, gpu)
    print("prefill_t512 dispatch", run_case(synth.GLM_LAYER, 512, seed=1, device=gpu,
                                            sample=[3, 200, 509]))


def test_fused_workspace_shared_across_descs_and_calls(gpu):
    """One workspace serves fused calls of different E in any order: the counters
    the kernel carries between calls (a call-counting barrier) never overlap
    another call's readiness counters, so every result equals the one on a fresh
    workspace."""
    from routed_expert_decode_gb300 import moe

    specs = [_spec(E=64, k=4, d=512, f=256, f_shared=256, s=2.5, zipf_beta=0.4),
             _spec(E=16, k=4, d=256, f=256, f_shared=0)]
    layers = [device_layer(s, gpu) for s in specs[:1]]
    ws = torch.zeros(1 << 24, dtype=torch.uint8, device=gpu)
    order = [0, 1, 0, 0, 1, 1, 0]
    for call, i in enumerate(order):
        spec = specs[i]
        layer = device_layer(spec, gpu)  # one resident layer at a time
        assert moe.layer_path(layer.desc(), 1) == "fused_decode"
        logits, x = synth.token_inputs(spec, 40 + call, 1)
        args = [torch.from_numpy(a).to(gpu) for a in (x, logits, synth.bias(spec))]
        y = torch.empty((1, spec.d), dtype=torch.float32, device=gpu)
        y_ref = torch.empty_like(y)
        moe.layer(layer.desc(), layer.weights, *args, y, ws)
        fresh = torch.zeros(moe.workspace_size(layer.desc(), 1), dtype=torch.uint8, device=gpu)
        moe.layer(layer.desc(), layer.weights, *args, y_ref, fresh)
        torch.cuda.synchronize()
        assert moe.check_device_error(ws) == 0
        assert torch.equal(y, y_ref), f"call {call} (E={spec.E})"
    del layers


@pytest.mark.parametrize("T", [8, 16, 64])
def test_tensor_core_dispatch_needs_a_tile_per_sm(gpu, T):
    """Auto dispatch on the full layer: the tensor-core path is taken only when
    the experts above the row threshold bring at least one gate/up tile per SM
    (else every expert runs on the GEMV); the plan's tensor-expert count agrees
    with the rule restated on the host, and the output matches the oracle."""
    import os
    import sys

    from routed_expert_decode_gb300 import moe

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    spec = synth.GLM_LAYER
    layer = device_layer(spec, gpu)
    rep = run_case(spec, T, seed=2, device=gpu, sample=[0, T - 1], check_taps=False)
    ws = layer.workspace(T, 0)
    L = moe.workspace_layout(layer.desc(), T)
    hdr = ws[L.plan:L.plan + 32].view(torch.int32).cpu().tolist()
    off = layer.views(ws, T)["off"].cpu().numpy()
    counts = (off[1:] - off[:-1]).tolist()
    sms = torch.cuda.get_device_properties(gpu).multi_processor_count
    thr = moe.tc_min_rows(layer.desc(), T)
    want_tc = thr is not None and thr >= 0 and bench.tc_tiles(spec, T, counts, thr) >= sms
    assert (hdr[5] > 0) == want_tc, (T, hdr[5], bench.tc_tiles(spec, T, counts, thr), sms)
    print("dispatch", T, hdr[5], rep)


def test_tensor_core_plan_lists_widest_experts_first(gpu):
    """The plan's tensor-core list (the order the tensor kernels deal tiles out
    in) holds exactly the experts with rows plus the shared expert, sorted by
    rows, descending, the lower expert index first on equal rows; each entry's
    first slot and rows agree with the routing offsets, and the tile prefixes
    count (f/128) x ceil(rows/64) gate/up and (d/128) x ceil(rows/64) down tiles
    per entry in that order."""
    from routed_expert_decode_gb300 import moe

    spec = _spec(E=32, k=4, d=512, f=256, f_shared=256, s=2.5, zipf_beta=0.4)
    T, E = 64, 32
    fl = moe.FLAG_FORCE_TC
    layer = device_layer(spec, gpu)
    logits, x = synth.token_inputs(spec, 5, T)
    out = layer.forward(torch.from_numpy(x).to(gpu), torch.from_numpy(logits).to(gpu),
                        torch.from_numpy(synth.bias(spec)).to(gpu), flags=fl)
    torch.cuda.synchronize()
    ws = layer.workspace(T, fl)
    L = moe.workspace_layout(layer.desc(fl), T)
    n_int = 8 + 9 * (E + 2)
    plan = ws[L.plan:L.plan + 4 * n_int].view(torch.int32).cpu().numpy()
    item_gu = 8 + 3 * (E + 1)
    tc_e = item_gu + (E + 2)
    tc_row0, tc_rows = tc_e + (E + 1), tc_e + 2 * (E + 1)
    tc_tile_gu = tc_e + 3 * (E + 1)
    tc_tile_dn = tc_tile_gu + (E + 2)
    V = int(plan[5])
    off = out.off.cpu().numpy()
    rows_of = {e: int(off[e + 1] - off[e]) for e in range(E) if off[e + 1] > off[e]}
    rows_of[E] = T
    es = [int(v) for v in plan[tc_e:tc_e + V]]
    rows = [int(v) for v in plan[tc_rows:tc_rows + V]]
    assert sorted(es) == sorted(rows_of), (es, rows_of)
    assert rows == [rows_of[e] for e in es]
    for i in range(V - 1):
        assert rows[i] > rows[i + 1] or (rows[i] == rows[i + 1] and es[i] < es[i + 1]), (i, es, rows)
    R = T * spec.k
    assert [int(v) for v in plan[tc_row0:tc_row0 + V]] == [R if e == E else int(off[e]) for e in es]
    mt, dt = spec.f // 128, spec.d // 128
    gu, dn = 0, 0
    for i, r in enumerate(rows):
        assert plan[tc_tile_gu + i] == gu and plan[tc_tile_dn + i] == dn, i
        gu += mt * ((r + 63) // 64)
        dn += dt * ((r + 63) // 64)
    assert plan[tc_tile_gu + V] == gu == plan[6] and plan[tc_tile_dn + V] == dn == plan[7]


# ---------------------------------------------------------------- uninitialised-memory guard
POISON = [
    ("fused_t1", synth.GLM_LAYER_E32, 1, 0),
    ("fused_t2", synth.GLM_LAYER_E32, 2, 0),
    ("gemv_t16", synth.GLM_LAYER_E32, 16, 0),
    ("tc_forced_t40", _spec(E=16, k=4, d=512, f=256, f_shared=256, s=2.5, zipf_beta=0.4), 40, "tc"),
    ("tc_auto_t512", synth.GLM_LAYER_E32, 512, 0),
    ("q2_t13", _spec(E=192, k=8, d=512, f=192, f_shared=160, fmt=1, zipf_beta=0.4), 13, 0),
    ("fp4_t13", _spec(E=192, k=8, d=512, f=192, f_shared=160, fmt=2, zipf_beta=0.4), 13, 0),
    ("fp4_tc_t40", _spec(E=16, k=4, d=512, f=256, f_shared=256, fmt=2, s=1.0), 40, "tc"),
]


@pytest.mark.parametrize("name,spec,T,fl", POISON, ids=[p[0] for p in POISON])
def test_poisoned_workspace(gpu, name, spec, T, fl):
    """Every workspace byte past the fixed head set to 0xFF before the call: a
    kernel that reads scratch it has not written (the class of bug behind the
    pages' streaming regressions: NeutronStar glm-local README, "Latent
    CUDA-streaming bugs") would see NaN floats and out-of-range indices and fail
    parity.  Run twice, so the second call also starts from poison, not from the
    first call's leftovers."""
    from routed_expert_decode_gb300 import moe

    flags = moe.FLAG_FORCE_TC if fl == "tc" else 0
    sample = None if T <= 16 else [0, T // 2, T - 1]
    for seed in (31, 32):
        rep = run_case(spec, T, seed=seed, device=gpu, flags=flags, sample=sample, poison=True)
        print(name, seed, rep)
