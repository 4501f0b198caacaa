"""Pins of the oracle's QK-norm ("SageBwd: A Trainable Low-bit Attention" (structured summary),
"QK-norm": RMSNorm(x) = x / sqrt(mean x^2) * gamma; epsilon 1e-6) against things other than its
own formulas: finite differences, invariants and a hand-worked row."""
from __future__ import annotations

from fractions import Fraction as Fr

import numpy as np

import workloads
from oracle import qknorm


def _f64(x, g, eps):
    """y = g * x / sqrt(mean(x^2) + eps) in plain float64 (the definition, for differentiation)."""
    return g * x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)


def test_backward_matches_central_differences():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, 16)) * 2.0
    g = rng.uniform(0.5, 1.5, 16)
    w = rng.standard_normal((3, 16))
    eps = 1e-3
    r = 1.0 / np.sqrt((x * x).mean(axis=-1) + eps)
    dx, dg = qknorm.rms_norm_bwd(x, g, r, w)
    h = 1e-6
    num_dx = np.zeros_like(x)
    for i in range(x.shape[0]):
        for c in range(x.shape[1]):
            xp, xm = x.copy(), x.copy()
            xp[i, c] += h
            xm[i, c] -= h
            num_dx[i, c] = ((w * _f64(xp, g, eps)).sum() - (w * _f64(xm, g, eps)).sum()) / (2 * h)
    num_dg = np.zeros_like(g)
    for c in range(g.size):
        gp, gm = g.copy(), g.copy()
        gp[c] += h
        gm[c] -= h
        num_dg[c] = ((w * _f64(x, gp, eps)).sum() - (w * _f64(x, gm, eps)).sum()) / (2 * h)
    assert np.max(np.abs(dx - num_dx)) <= 1e-7 * np.max(np.abs(num_dx))
    assert np.max(np.abs(dg - num_dg)) <= 1e-7 * np.max(np.abs(num_dg))


def test_gradient_is_orthogonal_to_x_without_eps():
    """At eps = 0, gamma = 1 the norm is scale invariant, so sum_c dx_c x_c = 0."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((4, 64))
    r = 1.0 / np.sqrt((x * x).mean(axis=-1))
    dx, _ = qknorm.rms_norm_bwd(x, None, r, rng.standard_normal((4, 64)))
    assert np.max(np.abs((dx * x).sum(axis=-1))) <= 1e-12 * np.abs(dx).sum()


def test_power_of_two_scaling_is_exact():
    """Scaling a row by 2^k scales its sum of squares by 4^k exactly and r by 2^-k, so at eps = 0
    the normalised 16-bit values are bit-identical."""
    rng = np.random.default_rng(2)
    x = workloads.round_fp16(rng.standard_normal((8, 128)).astype(np.float32))
    y0, r0 = qknorm.rms_norm(x, None, 0.0, workloads.round_fp16)
    for k in (-6, 3):
        y1, r1 = qknorm.rms_norm(x * np.float32(2.0 ** k), None, 0.0, workloads.round_fp16)
        assert np.array_equal(y0, y1)
        assert np.array_equal(r1, r0 * np.float32(2.0 ** -k))


def test_hand_worked_row():
    """x = [3, 4, 0, 0]: mean square 25/4, eps 0 -> r = 0.4 rounded to float32, y = [1.2, 1.6, 0, 0]
    after the float32 products (then fp16: 1.2 -> 1.2001953125, 1.6 -> 1.599609375)."""
    x = np.array([[3.0, 4.0, 0.0, 0.0]], np.float32)
    y, r = qknorm.rms_norm(x, None, 0.0, workloads.round_fp16)
    assert r[0] == np.float32(0.4)
    assert y.tolist() == [[1.2001953125, 1.599609375, 0.0, 0.0]]
    y2, _ = qknorm.rms_norm(x, np.array([2.0, 0.5, 1.0, 1.0], np.float32), 0.0, workloads.round_fp16)
    assert y2.tolist() == [[2.400390625, 0.7998046875, 0.0, 0.0]]


def test_row_factor_is_the_correctly_rounded_exact_value():
    """r must be the float32 nearest to the exact 1 / sqrt(sum(x^2)/d + eps), eps the float32 value
    passed: with m_lo, m_hi the midpoints between r and its float32 neighbours,
    1/m_hi^2 < v < 1/m_lo^2 in exact rationals (v = the exact mean square + eps)."""
    rng = np.random.default_rng(3)
    eps = np.float32(1e-6)
    for scale in (1.0, 1e-3, 40.0):
        x = workloads.round_fp16((rng.standard_normal((100, 128)) * scale).astype(np.float32))
        r = qknorm.row_factor(x, eps)
        for row, rv in zip(x, r):
            v = sum(Fr(float(a)) ** 2 for a in row) / 128 + Fr(float(eps))
            lo = Fr(float(np.nextafter(rv, np.float32(0))))
            hi = Fr(float(np.nextafter(rv, np.float32(np.inf))))
            c = Fr(float(rv))
            m_lo, m_hi = (c + lo) / 2, (c + hi) / 2
            assert 1 / (m_hi * m_hi) < v < 1 / (m_lo * m_lo)
