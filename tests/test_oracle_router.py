"""Pins of the oracle's router front end (no GPU): spec-log1p, the DeepSeek
scoring sqrt(softplus(l)) ("256 experts, 512 lines", section "The constant that
always said 256": top-6, scale 1.5, E = 384) and the router logits GEMM (the
dot product of the fp32 inputs rounded once).  Each is checked against the mathematics -- libm in
fp64, closed forms, error bounds -- not against a retyped copy of itself."""
import math

import numpy as np
import pytest

import oracle
import refmath


def _ulp_err(got32, exact):
    got32 = np.asarray(got32, np.float32)
    ulp = np.spacing(np.abs(got32)).astype(np.float64)
    ulp = np.maximum(ulp, np.spacing(np.float32(np.finfo(np.float32).tiny)))
    return np.abs(got32.astype(np.float64) - exact) / ulp


def test_spec_log1p_accuracy():
    """log1p on [0, 1] within 3 ulp of libm: the series error (z^16/17 < 2^-26)
    plus roundings of z = y/(2+y), z^2, seven fmas and the final product."""
    rng = np.random.default_rng(3)
    y = np.concatenate([np.linspace(0.0, 1.0, 6001, dtype=np.float32),
                        (10.0 ** rng.uniform(-30, 0, 6000)).astype(np.float32),
                        np.float32([1e-38, 1e-20, 0.25, 0.5, 1.0])])
    got = oracle.spec_log1p(y)
    exact = np.array([math.log1p(float(v)) for v in y])
    err = _ulp_err(got, exact)
    assert err.max() <= 3.0, err.max()
    assert got[0] == 0.0  # log1p(0) = 0 exactly


def test_sqrt_softplus_accuracy_and_shape():
    """sqrt(softplus(l)) within 3 ulp of the fp64 formula over the logit range;
    value at 0 is sqrt(ln 2); non-decreasing; softplus(l) - softplus(-l) = l."""
    l = np.linspace(-60.0, 60.0, 24001, dtype=np.float32)
    got = oracle.sqrt_softplus(l)
    exact = np.array([math.sqrt(max(v, 0.0) + math.log1p(math.exp(-abs(v)))) for v in l.astype(np.float64)])
    assert _ulp_err(got, exact).max() <= 3.0
    assert abs(float(oracle.sqrt_softplus([0.0])[0]) - math.sqrt(math.log(2.0))) < 2 ** -23
    assert np.all(np.diff(got.astype(np.float64)) >= 0)
    sp_pos = got.astype(np.float64) ** 2
    sp_neg = oracle.sqrt_softplus(-l).astype(np.float64) ** 2
    assert np.allclose(sp_pos - sp_neg, l.astype(np.float64), atol=1e-4 * (1 + np.abs(l)))


def test_score_fn_sigmoid_matches_score():
    rng = np.random.default_rng(5)
    l = rng.normal(size=512).astype(np.float32)
    b = (rng.normal(size=512) * 0.1).astype(np.float32)
    p, c = oracle.score_fn(oracle.SCORE_SIGMOID, l, b)
    s, c2 = oracle.score(l, b)
    assert np.array_equal(p, s) and np.array_equal(c, c2)
    p2, c3 = oracle.score_fn(oracle.SCORE_SQRT_SOFTPLUS, l, b)
    assert np.array_equal(p2, oracle.sqrt_softplus(l))
    assert np.array_equal(c3, (p2 + b).astype(np.float32))


@pytest.mark.parametrize("s", [1.0, 1.5])
def test_route_sqrt_softplus_topk_and_weights(s):
    """DeepSeek-style routing, E=384, top-6: the picks are the brute-force top-k
    of sqrt(softplus(l)) + b; weights are s * p_j / sum p_j."""
    rng = np.random.default_rng(11)
    T, E, k = 32, 384, 6
    logits = rng.normal(size=(T, E)).astype(np.float32)
    bias = (rng.normal(size=E) * 0.1).astype(np.float32)
    idx, w = oracle.route(logits, bias, k, s, score=oracle.SCORE_SQRT_SOFTPLUS)
    for t in range(T):
        _, c = oracle.score_fn(oracle.SCORE_SQRT_SOFTPLUS, logits[t], bias)
        assert np.array_equal(idx[t], refmath.brute_topk(c, k))
        lt = logits[t, idx[t]].astype(np.float64)
        p = np.sqrt(np.maximum(lt, 0) + np.log1p(np.exp(-np.abs(lt))))
        assert np.allclose(w[t], s * p / p.sum(), rtol=2 ** -22, atol=0)
        assert abs(float(w[t].astype(np.float64).sum()) - s) <= k * 2 ** -23 * s


def _exact_dot(x, w):
    """The exact value of sum_i x_i w_i for fp32 inputs (math.fsum of products
    that are exact in double), as a Python float."""
    return math.fsum(float(a) * float(b) for a, b in zip(x.astype(np.float64), w.astype(np.float64)))


@pytest.mark.parametrize("T,E,d", [(1, 8, 64), (3, 37, 256), (2, 24, 6144)])
def test_router_logits_are_the_dot_rounded_once(T, E, d):
    """Against the exact dot (fsum): the oracle's logit is within half an fp32
    ulp of it plus the fp64 accumulation error (d * 2^-53 * sum|x_i w_i|), i.e.
    the exact value rounded once; in practice it equals fp32(exact) almost
    always (a double-rounding miss needs the fp64 sum within 2^-29 of a tie)."""
    rng = np.random.default_rng(T * 1000 + E)
    x = rng.normal(size=(T, d)).astype(np.float32)
    w = (rng.normal(size=(E, d)) / math.sqrt(d)).astype(np.float32)
    got = oracle.router_logits(x, w)
    same = 0
    for t in range(T):
        for e in range(E):
            ex = _exact_dot(x[t], w[e])
            mag = float(np.abs(x[t].astype(np.float64)) @ np.abs(w[e].astype(np.float64)))
            g = float(got[t, e])
            half_ulp = float(np.spacing(np.float32(abs(ex)))) / 2
            assert abs(g - ex) <= half_ulp + d * 2.0 ** -53 * mag + 1e-300, (t, e)
            same += g == float(np.float32(ex))
    assert same >= T * E - 1


def test_router_logits_closed_forms():
    """One-hot x picks a weight column exactly; integer-valued inputs sum exactly."""
    d, E = 128, 5
    rng = np.random.default_rng(2)
    w = rng.normal(size=(E, d)).astype(np.float32)
    for i in (0, 31, 32, 77, 127):
        x = np.zeros((1, d), np.float32)
        x[0, i] = 1.0
        assert np.array_equal(oracle.router_logits(x, w)[0], w[:, i])
    wi = rng.integers(-8, 9, size=(E, d)).astype(np.float32)
    xi = rng.integers(-8, 9, size=(3, d)).astype(np.float32)
    exact = (xi.astype(np.int64) @ wi.T.astype(np.int64)).astype(np.float64)
    assert np.array_equal(oracle.router_logits(xi, wi).astype(np.float64), exact)


def test_router_logits_cancellation_is_exact():
    """Large terms that cancel do not swallow small ones: 2^24 + 1 - 2^24 = 1
    (an fp32 running sum would give 0) wherever the terms sit, and 2^24 - 2^24
    plus thirty ones is 30."""
    d = 3072
    for i0, i1, i2 in ((0, 1024, 2048), (5, 6, 7), (2048, 0, 1024)):
        x = np.zeros((1, d), np.float32)
        w = np.zeros((1, d), np.float32)
        x[0, [i0, i1, i2]] = 1.0
        w[0, i0], w[0, i1], w[0, i2] = 2.0 ** 24, 1.0, -(2.0 ** 24)
        assert oracle.router_logits(x, w)[0, 0] == 1.0
    x = np.ones((1, 32), np.float32)
    w = np.ones((1, 32), np.float32)
    w[0, 0], w[0, 16] = 2.0 ** 24, -(2.0 ** 24)
    assert oracle.router_logits(x, w)[0, 0] == 30.0


def test_router_logits_products_are_not_rounded():
    """(1 + 2^-12)^2 = 1 + 2^-11 + 2^-24 is not an fp32 number; with a second
    product 2^-24 the exact dot is 1 + 2^-11 + 2^-23, which is.  Rounding the
    first product to fp32 (a tie, to even: 1 + 2^-11) before adding would give
    1 + 2^-11 instead."""
    a = np.float32(1.0 + 2.0 ** -12)
    b = np.float32(2.0 ** -12)
    x = np.array([[a, b]], np.float32)
    w = np.array([[a, b]], np.float32)
    want = np.float32(1.0 + 2.0 ** -11 + 2.0 ** -23)
    assert float(want) == 1.0 + 2.0 ** -11 + 2.0 ** -23
    assert oracle.router_logits(x, w)[0, 0] == want
