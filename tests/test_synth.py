"""The seeded input generator: determinism, ranges, fp16 rounding and the
workload calibration (no GPU)."""
import numpy as np
import pytest

import oracle
import synth


def test_f64_to_f16_matches_numpy_rounding():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.random(200000) * 2e-4,                       # the scale range
        np.exp(rng.uniform(-20, 11.5, 200000)),          # normals and subnormals
        np.array([65504.0, 65519.99, 65520.0, 2 ** -24, 2 ** -25, 1.5 * 2 ** -25, 0.0]),
    ])
    # halfway points between fp16 neighbours must round to even
    h = np.arange(0x0400, 0x7BFF, 97, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (h + np.nextafter(h.astype(np.float16), np.float16(np.inf)).astype(np.float64)) / 2
    vals = np.concatenate([vals, mids, -vals[:1000]])
    got = np.array([synth.f64_to_f16_bits(v) for v in vals], np.uint16)
    with np.errstate(over="ignore"):  # 65520 rounds to inf, as it should
        ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_streams_are_deterministic_and_distinct():
    a = synth.int8(0, 16, 1000)
    assert np.array_equal(a, synth.int8(0, 16, 1000))
    assert not np.array_equal(a, synth.int8(0, 17, 1000))
    assert not np.array_equal(a, synth.int8(1, 16, 1000))
    assert np.array_equal(synth.int8(0, 16, 100, first=900), a[900:])
    assert np.array_equal(synth.normal(3, 2, 50, first=10), synth.normal(3, 2, 60)[10:])


def test_int8_range_and_uniformity():
    a = synth.int8(0, 20, 2_000_000).astype(np.int64)
    assert a.min() == -127 and a.max() == 127
    counts = np.bincount(a + 127, minlength=255)
    assert counts.min() > 0.9 * counts.mean() and counts.max() < 1.1 * counts.mean()


def test_code2_uniform():
    c = synth.code2(0, 21, 400000)
    codes = np.stack([(c >> s) & 3 for s in (0, 2, 4, 6)]).ravel()
    counts = np.bincount(codes, minlength=4)
    assert np.all(np.abs(counts / counts.sum() - 0.25) < 0.005)


def test_scale_range():
    K = 6144
    s = synth.scale_f16(0, 17, 100000, synth.scale_denom(0, K)).astype(np.float64)
    lo, hi = 0.5 / (127 * np.sqrt(K)), 1.5 / (127 * np.sqrt(K))
    assert s.min() >= lo * (1 - 2 ** -11) and s.max() <= hi * (1 + 2 ** -11)


def test_normal_moments():
    z = synth.normal(5, 2, 400000).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    b = synth.normal(0, synth.STREAM_BIAS, 200000, 0.0, 0.1).astype(np.float64)
    assert abs(b.std() - 0.1) < 0.002


def test_zipf_offset_is_a_permuted_log_rank():
    off = synth.zipf_offset(0, 3, 256, 0.4)
    ranks = np.exp(-off.astype(np.float64) / (0.4 * 1.1))
    assert np.allclose(np.sort(ranks), np.arange(1, 257), rtol=1e-5)


@pytest.mark.parametrize("spec", [synth.GLM_LAYER, synth.Q2_LAYER])
def test_zipf_workload_calibration(spec):
    """The popularity skew reproduces the pages' observations: the hottest ~4%
    of experts take ~30% of selections, two rows overlap ~10-20%."""
    logits, _ = synth.token_inputs(spec, 1234, 4000)
    idx, _ = oracle.route(logits, synth.bias(spec), spec.k, spec.s)
    counts = np.bincount(idx.ravel(), minlength=spec.E)
    top = int(round(0.04 * spec.E))
    share = np.sort(counts)[::-1][:top].sum() / counts.sum()
    assert 0.2 < share < 0.4, share
    overlap = np.mean([len(set(idx[2 * i]) & set(idx[2 * i + 1])) / spec.k
                       for i in range(2000)])
    assert 0.08 < overlap < 0.25, overlap
