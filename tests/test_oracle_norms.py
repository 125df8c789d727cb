"""Pins of the oracle's GroupNorm, RMS_norm and SiLU (CPU only).

GroupNorm: the printed two-group example, the closed form of the output
moments, invariance to a per-group affine change of x, and a brute-force
loop that fixes which channels form a group (consecutive, not interleaved).
RMS_norm: ||y|| = sqrt(C) for gamma = 1, a constant vector maps to
sign(a)*gamma, scale invariance, y(0) = 0, the bias added on read.
SiLU: SiLU(0) = 0, SiLU(v) - SiLU(-v) = v, and SiLU(1) = 1/(1+e^-1).
"""
import math

import numpy as np
import pytest

import oracle
from conftest import load_golden


def test_group_norm_printed_example():
    g = load_golden("group_norm_standardizes.json")
    x = np.array(g["x"], float)
    y = oracle.group_norm(x, g["groups"], np.array(g["gamma"]), np.array(g["beta"]), 1e-6)
    for p in g["printed"]:
        assert abs(y[p["c"], p["y"], p["x"]] - p["value"]) < p["tol"]
    assert abs(g["printed"][0]["value"] - (-3 / math.sqrt(5) * 2)) < 1e-15


@pytest.mark.parametrize("groups,c", [(32, 64), (4, 8), (2, 6)])
def test_group_norm_closed_form_moments(groups, c):
    rng = np.random.default_rng(11)
    x = rng.standard_normal((c, 5, 7)) * 3 + 2
    eps = 1e-6
    y = oracle.group_norm(x, groups, np.ones(c), np.zeros(c), eps)
    per = c // groups
    for g in range(groups):
        s = x[g * per:(g + 1) * per]
        t = y[g * per:(g + 1) * per]
        var = s.var()
        assert abs(t.mean()) < 1e-12
        assert abs(t.var() - var / (var + eps)) < 1e-12


def test_group_norm_per_group_affine_invariance():
    rng = np.random.default_rng(12)
    c, groups = 8, 4
    x = rng.standard_normal((c, 4, 4))
    gam, bet = rng.standard_normal(c), rng.standard_normal(c)
    a = np.repeat(rng.uniform(0.5, 2.0, groups), c // groups)[:, None, None]
    s = np.repeat(rng.standard_normal(groups), c // groups)[:, None, None]
    y1 = oracle.group_norm(x, groups, gam, bet, 0.0)
    y2 = oracle.group_norm(a * x + s, groups, gam, bet, 0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-10, atol=1e-10)


def test_group_norm_brute_force_membership_and_bias():
    rng = np.random.default_rng(13)
    c, groups, h, w = 6, 3, 2, 3
    x = rng.standard_normal((c, h, w))
    gam, bet, bi = rng.standard_normal((3, c))
    eps = 1e-6
    y = oracle.group_norm(x, groups, gam, bet, eps, bias_in=bi)
    per = c // groups
    for ch in range(c):
        g = ch // per
        vals = [x[cc, i, j] + bi[cc] for cc in range(g * per, (g + 1) * per) for i in range(h) for j in range(w)]
        mu = sum(vals) / len(vals)
        var = sum((v - mu) ** 2 for v in vals) / len(vals)
        for i in range(h):
            for j in range(w):
                ref = (x[ch, i, j] + bi[ch] - mu) / math.sqrt(var + eps) * gam[ch] + bet[ch]
                assert abs(y[ch, i, j] - ref) < 1e-12


def test_rms_norm_unit_gamma_norm_is_sqrt_c():
    rng = np.random.default_rng(14)
    c = 144
    x = rng.standard_normal((c, 3, 4)) * 5
    y = oracle.rms_norm(x, np.ones(c))
    np.testing.assert_allclose(np.sqrt((y ** 2).sum(axis=0)), math.sqrt(c), rtol=1e-13)


def test_rms_norm_constant_vector_and_zero():
    c = 16
    gam = np.linspace(0.5, 2.0, c)
    for a in (3.0, -0.25):
        x = np.full((c, 1, 1), a)
        y = oracle.rms_norm(x, gam)
        np.testing.assert_allclose(y[:, 0, 0], np.sign(a) * gam, rtol=1e-14)
    assert np.array_equal(oracle.rms_norm(np.zeros((c, 2, 2)), gam), np.zeros((c, 2, 2)))


def test_rms_norm_scale_invariance_and_bias_on_read():
    rng = np.random.default_rng(15)
    c = 48
    x = rng.standard_normal((c, 2, 5))
    gam = rng.standard_normal(c)
    np.testing.assert_allclose(oracle.rms_norm(7.5 * x, gam), oracle.rms_norm(x, gam), rtol=1e-13)
    b = rng.standard_normal(c)
    np.testing.assert_allclose(oracle.rms_norm(x, gam, bias_in=b),
                               oracle.rms_norm(x + b[:, None, None], gam), rtol=1e-14)


def test_rms_norm_brute_force_pixel():
    rng = np.random.default_rng(16)
    c = 5
    x = rng.standard_normal((c, 2, 2))
    gam = rng.standard_normal(c)
    y = oracle.rms_norm(x, gam)
    for i in range(2):
        for j in range(2):
            n = math.sqrt(sum(x[k, i, j] ** 2 for k in range(c)))
            for k in range(c):
                assert abs(y[k, i, j] - x[k, i, j] * math.sqrt(c) / n * gam[k]) < 1e-13


def test_silu_closed_forms():
    v = np.linspace(-30, 30, 121)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(oracle.silu(v) - oracle.silu(-v), v, rtol=1e-13, atol=1e-13)
    assert abs(oracle.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert oracle.silu(np.array([-1000.0]))[0] == 0.0
