"""Pins for the oracle's K/V-append step (RMS norm + rotate-half RoPE).

Checked against closed forms and invariants: a constant vector normalises to
the weight (up to eps); position 0 is the plain RMS norm; a one-hot input at
dim i rotates by exactly pos * theta^(-i/64) into dims (i, i+64) (for i = 32,
theta = 1e6, pos = 1000 the angle is exactly 1 rad); the norm is invariant to
positive scaling of x when eps = 0; the rotation preserves the vector norm;
and RoPE's relative-position property <z_q(m), z_k(n)> = <z_q(m+d), z_k(n+d)>.
test_oracle_mutants.py plants mistakes (interleaved pairs, a flipped sign, a
doubled frequency, sum instead of mean, eps dropped) and requires these pins
to catch them.
"""
import math

import numpy as np
import pytest

import oracle


def _nr(lib, x, w, pos, eps=1e-6, theta=1e6):
    return oracle.norm_rope(x, w, pos, eps, theta, lib)


def test_constant_vector_normalises_to_the_weight(orc):
    w = np.linspace(0.5, 1.5, 128)
    for c in (3.0, -0.25):
        z = _nr(orc, np.full(128, c), w, 0, eps=1e-6)
        np.testing.assert_allclose(z, np.sign(c) * w / math.sqrt(1 + 1e-6 / c ** 2), rtol=1e-14)


def test_position_zero_is_the_plain_rms_norm(orc):
    rng = np.random.default_rng(1)
    x, w = rng.standard_normal(128), rng.standard_normal(128)
    ms = math.fsum(v * v for v in x) / 128
    np.testing.assert_allclose(_nr(orc, x, w, 0, eps=0.01), x * w / math.sqrt(ms + 0.01), rtol=1e-13)


@pytest.mark.parametrize("i", [0, 1, 17, 32, 63])
def test_one_hot_rotates_into_its_rotate_half_partner(orc, i):
    pos, theta = 1000, 1e6
    x = np.zeros(128)
    x[i] = 1.0
    z = _nr(orc, x, np.ones(128), pos, eps=0.0, theta=theta)
    y = math.sqrt(128.0)  # a one-hot vector normalises to sqrt(d) at its dim
    a = pos * theta ** (-i / 64)
    want = np.zeros(128)
    want[i], want[i + 64] = y * math.cos(a), y * math.sin(a)
    np.testing.assert_allclose(z, want, rtol=1e-12, atol=1e-12)


def test_exact_one_radian_example(orc):
    # theta^(-32/64) = 1e-3 for theta = 1e6, so position 1000 turns dim 32 by 1 rad
    x = np.zeros(128)
    x[32] = 2.0
    z = _nr(orc, x, np.ones(128), 1000, eps=0.0, theta=1e6)
    assert z[32] == pytest.approx(math.sqrt(128) * 0.5403023058681398, rel=1e-12)
    assert z[96] == pytest.approx(math.sqrt(128) * 0.8414709848078965, rel=1e-12)
    assert np.count_nonzero(np.abs(z) > 1e-12) == 2


def test_norm_is_scale_invariant_without_eps(orc):
    rng = np.random.default_rng(2)
    x, w = rng.standard_normal(128), rng.standard_normal(128)
    np.testing.assert_allclose(_nr(orc, 37.5 * x, w, 123, eps=0.0), _nr(orc, x, w, 123, eps=0.0), rtol=1e-12)


def test_rotation_preserves_the_norm(orc):
    rng = np.random.default_rng(3)
    x, w = rng.standard_normal(128), rng.standard_normal(128)
    y = _nr(orc, x, w, 0)
    for pos in (1, 77, 131071):
        assert np.linalg.norm(_nr(orc, x, w, pos)) == pytest.approx(np.linalg.norm(y), rel=1e-12)


def test_relative_position_property(orc):
    rng = np.random.default_rng(4)
    xq, xk, w = rng.standard_normal(128), rng.standard_normal(128), np.ones(128)
    for m, n, d in ((5, 2, 40), (1000, 17, 4096), (0, 300, 1)):
        a = np.dot(_nr(orc, xq, w, m), _nr(orc, xk, w, n))
        b = np.dot(_nr(orc, xq, w, m + d), _nr(orc, xk, w, n + d))
        assert a == pytest.approx(b, rel=1e-9, abs=1e-9)
