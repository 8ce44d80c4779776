"""Pins for the oracle's RoPE.

The MTraining review (section on the Vertical-Slash pattern) states the
expected attention score of RoPE'd vectors as
  E[z_{n,m}] = sum_i phi^{(i)}_{n-m} A_i + sum_i psi^{(i)}_{n-m} B_i,
  phi^{(i)}_k = cos(k theta_{i mod d/2}),
  psi^{(i)}_k = (-1)^{[i >= d/2]} sin(k theta_{i mod d/2}),
  theta_i = 10000^{-2i/d},
with A_i, B_i position-free.  For fixed vectors the expectation is the score
itself with A_i = q_i k_i and B_i = q_i k_{(i + d/2) mod d}; that identity
fixes the rotate-half pairing and the sign of the sine terms.
"""
import math

import numpy as np
import pytest

from oracle import rope, rope_inv_freq, rope_mscale


def _rot(x, t, theta=1e4, **kw):
    return rope(x[None, None, :], theta, positions=np.array([t]), **kw)[0, 0]


@pytest.mark.parametrize("d", [8, 64, 128])
def test_expectation_equation_fixes_convention(d):
    rng = np.random.default_rng(d)
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    h = d // 2
    for n, m in [(5, 2), (100, 99), (4096, 17), (3, 3)]:
        lhs = _rot(q, n) @ _rot(k, m)
        rhs = 0.0
        for i in range(d):
            th = 10000.0 ** (-2.0 * (i % h) / d)
            phi = math.cos((n - m) * th)
            psi = (-1.0 if i >= h else 1.0) * math.sin((n - m) * th)
            rhs += phi * q[i] * k[i] + psi * q[i] * k[(i + h) % d]
        assert abs(lhs - rhs) < 1e-9 * (1 + abs(rhs))


def test_wrong_convention_is_caught():
    # interleaved-pair RoPE (channel 2i with 2i+1) breaks the identity above
    d, h = 8, 4
    rng = np.random.default_rng(0)
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    n, m = 7, 2
    def inter(x, t):
        y = x.copy()
        for i in range(h):
            th = 10000.0 ** (-2.0 * i / d)
            c, s = math.cos(t * th), math.sin(t * th)
            y[2 * i], y[2 * i + 1] = x[2 * i] * c - x[2 * i + 1] * s, x[2 * i + 1] * c + x[2 * i] * s
        return y
    rhs = sum(math.cos((n - m) * 10000.0 ** (-2.0 * (i % h) / d)) * q[i] * k[i]
              + (-1.0 if i >= h else 1.0) * math.sin((n - m) * 10000.0 ** (-2.0 * (i % h) / d)) * q[i] * k[(i + h) % d]
              for i in range(d))
    assert abs(inter(q, n) @ inter(k, m) - rhs) > 1e-3
    assert abs(_rot(q, n) @ _rot(k, m) - rhs) < 1e-9


def test_relative_position_and_norm():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 2, 32))
    y = rope(x, 1e4)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    q, k = rng.standard_normal(32), rng.standard_normal(32)
    for c in (1, 17, 1000):
        a = _rot(q, 40) @ _rot(k, 9)
        b = _rot(q, 40 + c) @ _rot(k, 9 + c)
        assert abs(a - b) < 1e-9


def test_transpose_inverts():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((50, 3, 16))
    np.testing.assert_allclose(rope(rope(x, 1e4), 1e4, transpose=True), x, atol=1e-12)
    # adjoint: <R x, y> == <x, R^T y>
    y = rng.standard_normal(x.shape)
    a = (rope(x, 5e5, yarn_factor=32, yarn_orig_len=16) * y).sum()
    b = (x * rope(y, 5e5, transpose=True, yarn_factor=32, yarn_orig_len=16)).sum()
    assert abs(a - b) < 1e-9 * abs(a)


def test_rotation_angle_closed_form():
    # first channel pair rotates by exactly t radians (theta_0 = 1)
    x = np.zeros((1, 1, 4)); x[0, 0, 0] = 1.0
    for t in (1, 3, 1000):
        y = rope(x, 1e4, positions=np.array([t]))[0, 0]
        np.testing.assert_allclose([y[0], y[2]], [math.cos(t), math.sin(t)], atol=1e-12)


def test_yarn_limits():
    d, base = 128, 5e5
    f0 = rope_inv_freq(d, base)
    np.testing.assert_array_equal(rope_inv_freq(d, base, 1.0, 4096), f0)
    s, orig = 32.0, 16384
    f = rope_inv_freq(d, base, s, orig)
    r = orig * f0 / (2 * math.pi)
    hi, lo = r >= 32.0, r <= 1.0
    assert hi.any() and lo.any()
    np.testing.assert_allclose(f[hi], f0[hi], rtol=1e-15)
    np.testing.assert_allclose(f[lo], f0[lo] / s, rtol=1e-15)
    mid = ~(hi | lo)
    assert np.all(f[mid] < f0[mid]) and np.all(f[mid] > f0[mid] / s)
    assert abs(rope_mscale(32.0) - (0.1 * math.log(32.0) + 1.0)) < 1e-15
    assert rope_mscale(1.0) == 1.0
