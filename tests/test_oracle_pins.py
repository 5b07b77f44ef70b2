"""Pins of the CPU oracle against facts outside itself (no GPU).

Each test checks one oracle function against a closed form, a textbook
definition, a brute-force computation or an invariant, chosen so that a
plausible slip (dropped term, wrong sign or index, transposed operand, swapped
gate/up, unstable permutation) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
import refmath
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ fp16 / spec-exp
def test_f16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def _ulp_err(got32: np.ndarray, exact: np.ndarray) -> np.ndarray:
    ulp = np.spacing(np.abs(got32.astype(np.float32))).astype(np.float64)
    return np.abs(got32.astype(np.float64) - exact) / ulp


def test_spec_exp_accuracy_sampled():
    """spec-exp against libm exp in fp64 over ~1M evenly spread fp32 inputs in
    [-86, 88]: at most 2 ulp (Cody-Waite + degree-7 Taylor error budget)."""
    lo = np.float32(-86.0).view(np.uint32)
    hi = np.float32(88.0).view(np.uint32)
    neg = np.arange(np.uint32(0x80000000), lo, 4096, dtype=np.uint64).astype(np.uint32)
    pos = np.arange(0, hi, 2048, dtype=np.uint64).astype(np.uint32)
    x = np.concatenate([neg, pos]).view(np.float32)
    got = oracle.spec_exp(x)
    err = _ulp_err(got, np.exp(x.astype(np.float64)))
    assert err.max() <= 2.0, f"max ulp error {err.max()}"
    # dense sweep where router/SiLU arguments live
    x2 = np.linspace(-12, 12, 400001, dtype=np.float32)
    err2 = _ulp_err(oracle.spec_exp(x2), np.exp(x2.astype(np.float64)))
    assert err2.max() <= 2.0


def test_spec_exp_special_points():
    got = oracle.spec_exp(np.array([0.0, -0.0, 1e-30, -1e3, 1e3, -86.0, 88.0], np.float32))
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == 1.0
    assert got[3] == oracle.spec_exp([-86.0])[0]   # clamped below
    assert got[4] == oracle.spec_exp([88.0])[0]    # clamped above
    assert np.isfinite(got).all() and (got > 0).all()


# ------------------------------------------------------------------ A1/A2 routing
def test_score_is_sigmoid_plus_bias():
    rng = np.random.default_rng(1)
    l = rng.normal(size=4096).astype(np.float32) * 4
    b = rng.normal(size=4096).astype(np.float32) * 0.1
    sigma, c = oracle.score(l, b)
    exact = refmath.sigmoid64(l)
    assert np.max(np.abs(sigma - exact) / exact) < 4 * 2 ** -24
    # the selection score is sigma + bias rounded once to fp32
    assert np.array_equal(c, (sigma + b).astype(np.float32))


@pytest.mark.parametrize("E,k", [(4, 1), (8, 3), (16, 4), (16, 16), (37, 8), (256, 8)])
def test_topk_matches_full_sort(E, k):
    rng = np.random.default_rng(E * 100 + k)
    for trial in range(50):
        l = rng.normal(size=E).astype(np.float32)
        # quantise logits so that exact score ties occur often
        if trial % 2:
            l = np.round(l * 2) / 2
        b = (rng.normal(size=E) * 0.1).astype(np.float32)
        if trial % 3 == 0:
            b[:] = 0
        _, c = oracle.score(l, b)
        assert np.array_equal(oracle.topk(c, k), refmath.brute_topk(c, k))


def test_topk_ties_take_lower_index():
    c = np.full(16, 0.5, np.float32)
    assert list(oracle.topk(c, 4)) == [0, 1, 2, 3]
    c[[3, 9, 12]] = 0.75
    assert list(oracle.topk(c, 5)) == [3, 9, 12, 0, 1]


def test_topk_all_selected_when_k_equals_E():
    rng = np.random.default_rng(3)
    c = rng.normal(size=16).astype(np.float32)
    idx = oracle.topk(c, 16)
    assert sorted(idx) == list(range(16))
    assert np.all(np.diff(c[idx]) <= 0)


@pytest.mark.parametrize("s", [1.0, 1.5, 2.5])
def test_route_weights_sum_to_scale_and_follow_sigmoid(s):
    rng = np.random.default_rng(7)
    T, E, k = 64, 256, 8
    logits = rng.normal(size=(T, E)).astype(np.float32)
    bias = (rng.normal(size=E) * 0.1).astype(np.float32)
    idx, w = oracle.route(logits, bias, k, s)
    for t in range(T):
        assert len(set(idx[t])) == k and idx[t].min() >= 0 and idx[t].max() < E
        _, c = oracle.score(logits[t], bias)
        assert np.array_equal(idx[t], refmath.brute_topk(c, k))
        sg = refmath.sigmoid64(logits[t, idx[t]])
        assert np.allclose(w[t], s * sg / sg.sum(), rtol=2 ** -23, atol=0)
        assert abs(float(w[t].astype(np.float64).sum()) - s) <= k * 2 ** -23 * s


def test_bias_changes_selection_not_weights():
    """The bias steers selection only: weights use sigmoid(logit) alone."""
    l = np.array([0.0, 0.1, 0.2, 0.3], np.float32)
    b = np.array([1.0, 0.0, 0.0, 0.0], np.float32)
    idx, w = oracle.route(l[None], b, 2, 1.0)
    assert list(idx[0]) == [0, 3]
    sg = refmath.sigmoid64(l[[0, 3]])
    assert np.allclose(w[0], sg / sg.sum(), rtol=1e-7)


# ------------------------------------------------------------------ A3 permutation
@pytest.mark.parametrize("T,E,k", [(1, 256, 8), (4, 16, 4), (16, 256, 8), (512, 256, 8),
                                   (7, 5, 5), (3, 1024, 1)])
def test_permutation_invariants(T, E, k):
    rng = np.random.default_rng(T + E + k)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    off, perm, pos = oracle.permute(idx, E)
    assert refmath.check_permutation(idx, off, perm, pos, E) == []
    roff, rperm, rpos = refmath.stable_permutation(idx, E)
    assert np.array_equal(off, roff) and np.array_equal(perm, rperm)
    assert np.array_equal(pos, rpos)


def test_permutation_checker_rejects_planted_mistake():
    """Negative control: a swapped pair in the oracle's permutation must fail."""
    rng = np.random.default_rng(5)
    idx = np.stack([rng.choice(16, size=4, replace=False) for _ in range(8)]).astype(np.int32)
    off, perm, pos = oracle.permute(idx, 16)
    bad = perm.copy()
    e = int(np.argmax(np.diff(off)))  # an expert with >= 2 rows
    a, b = off[e], off[e] + 1
    bad[a], bad[b] = bad[b], bad[a]
    assert refmath.check_permutation(idx, off, bad, pos, 16) != []


# ------------------------------------------------------------------ A4 quantisation
def _load_quant_cases():
    cases = []
    with open(os.path.join(GOLDEN, "quantize_hand_cases.txt")) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            xs, qs, sc = line.split("|")
            cases.append(([float(v) for v in xs.split()], [int(v) for v in qs.split()],
                          float.fromhex(sc.strip())))
    return cases


def test_quantize_hand_cases():
    for x_head, q_head, scale in _load_quant_cases():
        x = np.zeros(32, np.float32)
        x[:len(x_head)] = x_head
        q, sc = oracle.quantize(x)
        assert sc[0] == np.float32(scale), (x_head, sc[0], scale)
        assert list(q[:len(q_head)]) == q_head, (x_head, list(q[:len(q_head)]))
        assert np.all(q[len(q_head):] == 0)


def test_quantize_matches_textbook_definition():
    rng = np.random.default_rng(11)
    x = rng.normal(size=32 * 20000).astype(np.float32)
    x[:32] = 0
    x[32:64] *= 1e-30
    q, sc = oracle.quantize(x)
    rq, rsc = refmath.quantize(x)
    assert np.array_equal(sc, rsc)
    assert np.array_equal(q, rq)
    assert q.min() >= -127 and q.max() <= 127
    # the element reaching max|x| in each block maps to +-127
    blocks = x.reshape(-1, 32)[1:]
    am = np.abs(blocks).argmax(axis=1)
    qb = q.reshape(-1, 32)[1:]
    assert np.all(np.abs(qb[np.arange(len(am)), am]) == 127)


# ------------------------------------------------------------------ A10 2-bit
def test_decode_q2_mapping_and_order():
    # byte 0b11_10_01_00 holds codes 0,1,2,3 for weights 0..3 (LSB first)
    assert list(oracle.decode_q2(np.array([0b11100100], np.uint8), 4)) == [-3, -1, 1, 3]
    assert list(oracle.decode_q2(np.array([0x00], np.uint8), 4)) == [-3] * 4
    assert list(oracle.decode_q2(np.array([0xFF], np.uint8), 4)) == [3] * 4
    codes = synth.code2(0, 99, 64)
    assert np.array_equal(oracle.decode_q2(codes, 256), refmath.decode_q2(codes, 256))


# ------------------------------------------------------------------ 4-bit e2m1
def test_decode_e2m1_table_and_order():
    """The e2m1 value set (OCP microscaling FP4: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and
    their negatives, sign in bit 3), decoded as twice the value; low nibble
    first.  Pinned against the table and against numpy's float16 decoding of
    the same sign / exponent / mantissa fields."""
    nib = np.arange(16, dtype=np.uint8)
    packed = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)  # codes 0..15 in order
    got = oracle.decode_e2m1(packed, 16).astype(np.float64) / 2
    table = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(got[:8]) == table and list(got[8:]) == [-v for v in table]
    assert list(oracle.decode_e2m1(np.array([0x71], np.uint8), 2)) == [1, 12]  # low nibble first
    codes = synth.code2(0, 98, 512)
    assert np.array_equal(oracle.decode_e2m1(codes, 1024).astype(np.float64) / 2,
                          refmath.decode_e2m1_value(codes, 1024))


def test_matvec_e2m1_halves_the_doubled_dots():
    """Rows of code 2 (the value 1.0) with scale 1: g = sum of the activations,
    x codes times their scales, exactly; the block dots are of twice the values."""
    K = 128
    rng = np.random.default_rng(23)
    xq = rng.integers(-127, 128, size=K).astype(np.int8)
    xs = (rng.random(K // 32) + 0.5).astype(np.float32)
    wq = np.full((3, K // 2), 0x22, np.uint8)
    ws = np.full((3, K // 32), np.float16(1.0))
    want = float((xq.astype(np.float64) * np.repeat(xs.astype(np.float64), 32)).sum())
    assert np.array_equal(oracle.matvec(2, wq, ws, xq, xs), np.full(3, want))
    dots = oracle.block_dots(2, K, wq[0], xq)
    assert np.array_equal(dots, 2 * xq.astype(np.int32).reshape(-1, 32).sum(axis=1))


# ------------------------------------------------------------------ A5/A7 block dots
@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_block_dots_vs_int64(fmt):
    rng = np.random.default_rng(13 + fmt)
    K = 6144
    xq = rng.integers(-127, 128, size=K).astype(np.int8)
    if fmt == 0:
        w = rng.integers(-127, 128, size=K).astype(np.int8)
        wi = w.astype(np.int64)
    elif fmt == 1:
        w = rng.integers(0, 256, size=K // 4).astype(np.uint8)
        wi = refmath.decode_q2(w, K).astype(np.int64)
    else:  # twice the e2m1 values, from numpy's float16 decoding
        w = rng.integers(0, 256, size=K // 2).astype(np.uint8)
        wi = (2 * refmath.decode_e2m1_value(w, K)).astype(np.int64)
    got = oracle.block_dots(fmt, K, w, xq)
    ref = (wi * xq.astype(np.int64)).reshape(-1, 32).sum(axis=1)
    assert np.array_equal(got.astype(np.int64), ref)


def test_block_dot_extremes_fit_int32():
    K = 64
    w = np.full(K, -127, np.int8)
    xq = np.full(K, -127, np.int8)
    assert list(oracle.block_dots(0, K, w, xq)) == [32 * 127 * 127] * 2


def test_matvec_one_hot_rows_pick_single_activation():
    """Row n has a single 1 at column n (scale 1.0): g_n = xq[n] * xs[n // 32] exactly."""
    K = 128
    rng = np.random.default_rng(17)
    xq = rng.integers(-127, 128, size=K).astype(np.int8)
    xs = (rng.random(K // 32) + 0.5).astype(np.float32)
    wq = np.eye(K, dtype=np.int8)
    ws = np.full((K, K // 32), np.float16(1.0))
    g = oracle.matvec(0, wq, ws, xq, xs)
    assert np.array_equal(g, xq.astype(np.float64) * np.repeat(xs.astype(np.float64), 32))


def test_matvec_all_ones_gives_block_sums_times_scales():
    K = 256
    rng = np.random.default_rng(19)
    xq = rng.integers(-127, 128, size=K).astype(np.int8)
    xs = (rng.random(K // 32) + 0.5).astype(np.float32)
    ws = rng.random((3, K // 32)).astype(np.float16) + np.float16(0.25)
    wq = np.ones((3, K), np.int8)
    g = oracle.matvec(0, wq, ws, xq, xs)
    bsum = xq.astype(np.int64).reshape(-1, 32).sum(axis=1).astype(np.float64)
    ref = (ws.astype(np.float64) * xs.astype(np.float64)[None, :] * bsum[None, :]).sum(axis=1)
    assert np.allclose(g, ref, rtol=1e-15, atol=0)


# ------------------------------------------------------------------ expert + layer
def _spec(**kw):
    base = dict(name="t", E=16, k=4, d=256, f=128, f_shared=0, fmt=0, s=1.0, zipf_beta=0.0)
    base.update(kw)
    return synth.LayerSpec(**base)


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_expert_row_matches_dense_fp64(fmt):
    spec = _spec(fmt=fmt, d=512, f=256)
    ex = synth.expert_host(spec, 3)
    _, x = synth.token_inputs(spec, 1, 1)
    xq, xs = oracle.quantize(x[0])
    hq, hs, o = oracle.expert_row(fmt, spec.d, spec.f, ex, xq, xs)
    rhq, rhs, ro = refmath.expert_ffn(ex, fmt, spec.d, spec.f, xq, xs)
    flips = np.abs(hq.astype(int) - rhq.astype(int))
    assert flips.max() <= 1 and (flips > 0).mean() < 1e-2
    if flips.max() == 0:
        assert np.array_equal(hs, rhs)
        assert np.max(np.abs(o - ro)) <= 1e-12 * np.max(np.abs(ro))


def test_expert_row_detects_swapped_gate_up():
    """Negative control: an oracle with gate and up swapped disagrees with the
    dense re-derivation (SiLU makes the two roles asymmetric)."""
    spec = _spec()
    ex = synth.expert_host(spec, 0)
    swapped = dict(ex, gate_q=ex["up_q"], gate_s=ex["up_s"], up_q=ex["gate_q"], up_s=ex["gate_s"])
    _, x = synth.token_inputs(spec, 2, 1)
    xq, xs = oracle.quantize(x[0])
    _, _, o_bad = oracle.expert_row(0, spec.d, spec.f, swapped, xq, xs)
    _, _, ro = refmath.expert_ffn(ex, 0, spec.d, spec.f, xq, xs)
    assert np.max(np.abs(o_bad - ro)) > 1e-2 * np.max(np.abs(ro))


def _run_layer(spec, T, seed, want=None, drop_shared=False):
    logits, x = synth.token_inputs(spec, seed, T)
    bias = synth.bias(spec)
    experts = {e: synth.expert_host(spec, e) for e in range(spec.E)}
    shared = synth.expert_host(spec, spec.E) if spec.f_shared else None
    fs = 0 if drop_shared else spec.f_shared
    res = oracle.layer(spec.E, spec.k, spec.d, spec.f, fs, spec.fmt, spec.s, experts, shared,
                       x, logits, bias, want=want, score=spec.score)
    return res, experts, shared, x, logits, bias


@pytest.mark.parametrize("spec", [
    _spec(),                                                  # the tiny layer
    _spec(E=24, k=6, d=320, f=96, f_shared=64, s=2.5, zipf_beta=0.4),
    _spec(E=12, k=3, d=256, f=128, f_shared=96, fmt=1, s=1.0),
    _spec(E=12, k=3, d=256, f=128, f_shared=96, fmt=2, s=1.0),     # 4-bit e2m1 experts
    _spec(E=40, k=6, d=256, f=128, f_shared=128, s=1.5, score=1),  # DeepSeek scoring
])
def test_layer_matches_dense_rederivation(spec):
    T = 6
    res, experts, shared, x, logits, bias = _run_layer(spec, T, 3)
    for t in range(T):
        _, c = oracle.score_fn(spec.score, logits[t], bias)
        assert np.array_equal(res.idx[t], refmath.brute_topk(c, spec.k))
    assert refmath.check_permutation(res.idx, res.off, res.perm, res.pos, spec.E) == []
    rq, rs = refmath.quantize(x)
    assert np.array_equal(res.xq.ravel(), rq) and np.array_equal(res.xs.ravel(), rs)
    y_ref = refmath.layer(spec.E, spec.k, spec.d, spec.f, spec.f_shared, spec.fmt, spec.s,
                          experts, shared, x, res.idx, logits, score=spec.score)
    err = np.abs(res.y - y_ref).max(axis=1) / np.abs(y_ref).max(axis=1)
    assert err.max() < 1e-5, err


def test_layer_k1_is_one_dense_ffn():
    """k = 1, s = 1, no shared expert: y is the selected expert's quantised SwiGLU FFN."""
    spec = _spec(k=1)
    res, experts, _, x, _, _ = _run_layer(spec, 3, 4)
    for t in range(3):
        xq, xs = refmath.quantize(x[t])
        _, _, o = refmath.expert_ffn(experts[int(res.idx[t, 0])], 0, spec.d, spec.f, xq, xs)
        assert np.max(np.abs(res.y[t] - o)) <= 1e-5 * np.max(np.abs(o))
        assert res.w[t, 0] == 1.0


def test_layer_shared_expert_adds_its_ffn():
    spec = _spec(f_shared=64, s=2.5)
    with_s, experts, shared, x, _, _ = _run_layer(spec, 3, 5)
    without, *_ = _run_layer(spec, 3, 5, drop_shared=True)
    for t in range(3):
        xq, xs = refmath.quantize(x[t])
        _, _, o_s = refmath.expert_ffn(shared, 0, spec.d, 64, xq, xs)
        diff = with_s.y[t].astype(np.float64) - without.y[t].astype(np.float64)
        assert np.max(np.abs(diff - o_s)) <= 1e-5 * np.max(np.abs(with_s.y[t]))


def test_layer_all_experts_selected_when_k_equals_E():
    spec = _spec(E=6, k=6, d=128, f=64)
    res, *_ = _run_layer(spec, 4, 6)
    for t in range(4):
        assert sorted(res.idx[t]) == list(range(6))
    assert list(np.diff(res.off)) == [4] * 6


def test_layer_wanted_tokens_match_full_run():
    spec = _spec(E=32, k=4, f_shared=64)
    full, *_ = _run_layer(spec, 8, 9)
    part, *_ = _run_layer(spec, 8, 9, want=[1, 6])
    assert np.array_equal(full.y[[1, 6]], part.y[[1, 6]])
    assert np.isnan(part.y[0]).all()
    assert np.array_equal(full.idx, part.idx) and np.array_equal(full.off, part.off)


def test_layer_zero_tokens():
    spec = _spec()
    res, *_ = _run_layer(spec, 0, 0)
    assert res.y.shape == (0, spec.d)
    assert list(res.off) == [0] * (spec.E + 1)
