"""Pins for the oracle's layer arithmetic against closed forms and library routines (CPU)."""
import numpy as np
import pytest
import scipy.special

from oracle import dflash_oracle as orc


def test_rms_norm_hand_example():
    x = np.array([[3.0, 4.0]])
    y = orc.rms_norm(x, np.ones(2), 0.0)
    r = np.sqrt(12.5)
    assert np.allclose(y, [[3.0 / r, 4.0 / r]], rtol=0, atol=1e-15)
    # gain multiplies channel-wise
    y2 = orc.rms_norm(x, np.array([2.0, -1.0]), 0.0)
    assert np.allclose(y2, [[6.0 / r, -4.0 / r]], rtol=0, atol=1e-15)


def test_rms_norm_scale_invariance_and_unit_rms():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 64))
    g = np.ones(64)
    for c in (1e-3, 0.5, 7.0, 1e4):
        assert np.allclose(orc.rms_norm(c * x, g, 0.0), orc.rms_norm(x, g, 0.0), atol=1e-12)
    y = orc.rms_norm(x, g, 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-12)
    # eps matters only for tiny inputs
    assert np.allclose(orc.rms_norm(np.zeros((1, 4)), np.ones(4), 1e-6), 0.0)


def _rope_complex(x, positions, theta):
    """RoPE as complex multiplication: z_i = x_i + i x_{i+dh/2} times exp(i p theta^(-2i/dh))."""
    dh = x.shape[-1]
    half = dh // 2
    z = x[..., :half] + 1j * x[..., half:]
    freq = np.array([theta ** (-2.0 * i / dh) for i in range(half)])
    rot = np.exp(1j * np.outer(positions, freq))[:, None, :]
    w = z * rot
    return np.concatenate([w.real, w.imag], axis=-1)


@pytest.mark.parametrize("theta", [1e6, 1e4, 100.0])
def test_rope_equals_complex_rotation(theta):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 3, 8))
    pos = np.array([0, 1, 2, 17, 1000, 32767, 5])
    assert np.allclose(orc.apply_rope(x, pos, theta), _rope_complex(x, pos, theta), atol=1e-12)


def test_rope_identity_at_zero_and_norm_preserving():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 2, 128))
    assert np.array_equal(orc.apply_rope(x, np.zeros(4, int), 1e6), x)
    y = orc.apply_rope(x, np.array([3, 99, 4096, 32000]), 1e6)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), atol=1e-12)


def test_rope_relative_position_property():
    # <R(q, m), R(k, n)> depends only on m - n
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    def dot(m, n):
        return float(np.sum(orc.apply_rope(q, np.array([m]), 1e6) *
                            orc.apply_rope(k, np.array([n]), 1e6)))
    for m, n, t in [(5, 2, 100), (40, 41, 7), (0, 9, 3000)]:
        assert abs(dot(m, n) - dot(m + t, n + t)) < 1e-10
    # and it is not shift-free in a single argument (the rotation actually happens)
    assert abs(dot(5, 2) - dot(6, 2)) > 1e-6


def test_rope_first_pair_rotates_by_position():
    # channel pair (0, dh/2) has inverse frequency theta^0 = 1: rotation by p radians
    x = np.zeros((1, 1, 4))
    x[0, 0, 0] = 1.0
    y = orc.apply_rope(x, np.array([2]), 1e6)
    assert np.allclose(y[0, 0], [np.cos(2.0), 0.0, np.sin(2.0), 0.0], atol=1e-15)


def test_silu_closed_forms():
    x = np.linspace(-30, 30, 121)
    assert np.allclose(orc.silu(x), x * scipy.special.expit(x), atol=1e-14)
    assert orc.silu(np.array([0.0]))[0] == 0.0
    assert abs(orc.silu(np.array([40.0]))[0] - 40.0) < 1e-12


def test_softmax_against_library():
    rng = np.random.default_rng(4)
    s = rng.standard_normal((6, 11)) * 10
    assert np.allclose(orc.softmax_rows(s), scipy.special.softmax(s, axis=-1), atol=1e-15)
    assert np.allclose(orc.softmax_rows(s + 1234.5), orc.softmax_rows(s), atol=1e-15)
