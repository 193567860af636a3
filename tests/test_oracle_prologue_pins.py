"""Pins of the prologue oracle (QKV bias, YaRN rotary encoding, paged cache
write) to things other than itself (CPU only).

* hand-worked rotations in both pair layouts and a YaRN ramp midpoint
  (tests/golden/hand_examples.json);
* the rotation equals multiplication by exp(i p f) of the complex numbers
  x_a + i x_b (numpy complex arithmetic, a different route);
* relative position: <R(m) q, R(n) k> = mscale^2 <q, R(n - m) k> for any
  shift -- a sign or pairing mistake breaks it;
* factor 1 gives the plain frequencies base^(-2d/D) and magnitude 1; pairs
  outside the ramp are kept or divided by the factor exactly;
* the cache write touches exactly the mapped slots.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import prologue as pro

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def _golden(name):
    with open(GOLDEN) as f:
        return json.load(f)[name]


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_hand_rotation(style):
    c = _golden("rotary")
    x = np.array(c["x"])[None, None, :]
    out = pro.rotate(x, [1], [math.pi / 2, math.pi], 1.0, style)
    np.testing.assert_allclose(out[0, 0], c[style], atol=1e-14)
    out2 = pro.rotate(x, [1], [math.pi / 2, math.pi], 2.0, style)
    np.testing.assert_allclose(out2[0, 0], 2 * np.array(c[style]), atol=1e-14)


def test_hand_yarn_ramp_midpoint():
    c = _golden("yarn_ramp")
    f, m = pro.yarn_inv_freq(c["head_dim"], c["base"], c["factor"],
                             c["original_context_over_pi"] * math.pi, c["beta_fast"], c["beta_slow"])
    assert f.shape == (1,)
    assert abs(f[0] - 5 / 8) < 1e-15
    assert abs((m - 1) / math.log(4) - 0.1) < 1e-15


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_rotation_is_complex_multiplication(style):
    rng = np.random.default_rng(1)
    t, h, d = 7, 3, 64
    x = rng.standard_normal((t, h, d))
    pos = rng.integers(0, 200000, size=t)
    inv, ms = pro.yarn_inv_freq(d, 150000.0, 32.0, 4096, 32.0, 1.0)
    out = pro.rotate(x, pos, inv, ms, style)
    a, b = (np.arange(32), np.arange(32) + 32) if style == "half" else (np.arange(0, 64, 2), np.arange(1, 64, 2))
    z = (x[..., a] + 1j * x[..., b]) * (ms * np.exp(1j * np.outer(pos, inv)))[:, None, :]
    np.testing.assert_allclose(out[..., a], z.real, atol=1e-12)
    np.testing.assert_allclose(out[..., b], z.imag, atol=1e-12)


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_relative_position_property(style):
    rng = np.random.default_rng(2)
    d = 64
    inv, ms = pro.yarn_inv_freq(d, 10000.0, 8.0, 2048, 32.0, 1.0)
    for _ in range(20):
        q = rng.standard_normal((1, 1, d))
        k = rng.standard_normal((1, 1, d))
        m, n, shift = rng.integers(0, 5000, size=3)
        lhs = np.sum(pro.rotate(q, [m], inv, ms, style) * pro.rotate(k, [n], inv, ms, style))
        shifted = np.sum(pro.rotate(q, [m + shift], inv, ms, style) *
                         pro.rotate(k, [n + shift], inv, ms, style))
        rel = ms * ms * np.sum(q * pro.rotate(k, [n - m], inv, 1.0, style))
        np.testing.assert_allclose(lhs, shifted, rtol=1e-9, atol=1e-9)
        np.testing.assert_allclose(lhs, rel, rtol=1e-9, atol=1e-9)


def test_yarn_limits():
    d, base = 64, 150000.0
    f1, m1 = pro.yarn_inv_freq(d, base, 1.0, 4096, 32.0, 1.0)
    np.testing.assert_allclose(f1, base ** (-2.0 * np.arange(32) / d), rtol=1e-15)
    assert m1 == 1.0
    s = 32.0
    f, m = pro.yarn_inv_freq(d, base, s, 4096, 32.0, 1.0)
    theta = base ** (-2.0 * np.arange(32) / d)
    rot = 4096 * theta / (2 * math.pi)
    keep, scale = rot > 32.0, rot < 1.0
    assert keep.any() and scale.any()
    np.testing.assert_array_equal(f[keep], theta[keep])
    np.testing.assert_allclose(f[scale], theta[scale] / s, rtol=1e-15)
    assert np.all(np.diff(f) < 0)
    assert abs(m - (1 + 0.1 * math.log(32))) < 1e-15


def test_bias_then_rotation_and_v_unrotated():
    rng = np.random.default_rng(3)
    hq, hkv, d, t = 4, 2, 8, 5
    qkv = rng.standard_normal((t, (hq + 2 * hkv) * d))
    bias = rng.standard_normal((hq + 2 * hkv) * d)
    pos = np.arange(t) * 3
    inv, ms = pro.yarn_inv_freq(d, 500.0, 2.0, 64, 8.0, 1.0)
    q, k, v = pro.qkv_prologue(qkv, bias, pos, inv, ms, hq, hkv)
    x = (qkv + bias).reshape(t, hq + 2 * hkv, d)
    np.testing.assert_array_equal(v, x[:, hq + hkv:])
    np.testing.assert_allclose(q, pro.rotate(x[:, :hq], pos, inv, ms), atol=1e-15)
    np.testing.assert_allclose(k, pro.rotate(x[:, hq:hq + hkv], pos, inv, ms), atol=1e-15)
    # the norm of every pair grows by exactly the magnitude factor
    a, b = pro.pair_index(d, "half")
    np.testing.assert_allclose(np.hypot(q[..., a], q[..., b]),
                               ms * np.hypot(x[:, :hq, a], x[:, :hq, b]), rtol=1e-12)


def test_cache_scatter():
    cache = np.arange(3 * 2 * 4 * 2, dtype=np.float64).reshape(3, 2, 4, 2)
    vals = -np.ones((3, 2, 2)) * np.array([1, 2, 3])[:, None, None]
    out = pro.scatter_to_cache(cache, vals, [5, -1, 0], 4)
    expect = cache.copy()
    expect[1, :, 1] = vals[0]
    expect[0, :, 0] = vals[2]
    np.testing.assert_array_equal(out, expect)
