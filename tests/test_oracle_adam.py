"""Pins of the oracle's AdamW (Fudan MLSys ch. 9, 9.2.2, plus decoupled decay).

Closed forms that follow from the page's equations, not a retyping of them:
* first step from m = v = 0: m_hat = g, v_hat = g^2, so the update
  direction is g / (|g| + eps);
* a constant gradient for t steps from zero moments: m_t = (1 - b1^t) g and
  v_t = (1 - b2^t) g^2, so the bias corrections cancel exactly every step;
* b1 = b2 = 0: the moments are g and g^2 for any t (sign descent);
* g = 0 with zero moments leaves only the decoupled decay: w (1 - lr wd).
Each is sensitive to a dropped or swapped bias correction, epsilon under the
square root, a sign error, or decay applied after the Adam step.
"""

import numpy as np
import pytest


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.max(np.abs(a - b) / np.maximum(np.abs(b), 1e-30))


def test_first_step_closed_form(ora):
    rng = np.random.default_rng(0)
    n = 100_000
    g = (rng.standard_normal(n) * 10.0 ** rng.uniform(-6, 1, n)).astype(np.float32)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    lr, wd, eps = 0.1, 0.5, 1e-8
    w, m, v = ora.adamw(w0, np.zeros(n), np.zeros(n), g, lr, 0.9, 0.95, eps, wd, 1)
    gd = g.astype(np.float64)
    u = gd / (np.abs(gd) + eps)
    want = w0.astype(np.float64) * (1 - lr * wd) - lr * u
    assert np.max(np.abs(w - want)) < 5e-7
    assert _rel(m, 0.1 * gd) < 1e-6
    assert _rel(v, 0.05 * gd * gd) < 1e-6


def test_constant_gradient_closed_form(ora):
    rng = np.random.default_rng(1)
    n = 10_000
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    lr, wd, eps, b1, b2 = 0.01, 0.1, 1e-8, 0.9, 0.95
    want = w.astype(np.float64)
    gd = g.astype(np.float64)
    for t in range(1, 11):
        w, m, v = ora.adamw(w, m, v, g, lr, b1, b2, eps, wd, t)
        want = want * (1 - lr * wd) - lr * gd / (np.abs(gd) + eps)
        assert _rel(m, (1 - b1 ** t) * gd) < 1e-5
        assert _rel(v, (1 - b2 ** t) * gd * gd) < 1e-5
    assert np.max(np.abs(w - want)) < 1e-5


def test_sign_descent_when_betas_are_zero(ora):
    rng = np.random.default_rng(2)
    g = (rng.standard_normal(1000)).astype(np.float32)
    w0 = np.ones(1000, np.float32)
    m0 = rng.standard_normal(1000).astype(np.float32)
    v0 = rng.uniform(0, 1, 1000).astype(np.float32)
    for t in (1, 7):
        w, m, v = ora.adamw(w0, m0, v0, g, 0.25, 0.0, 0.0, 0.0, 0.0, t)
        assert np.array_equal(m, g)
        assert np.array_equal(v, g * g)
        assert np.array_equal(w, np.where(g > 0, 0.75, 1.25).astype(np.float32))


def test_zero_gradient_is_pure_decoupled_decay(ora):
    w0 = np.array([0.5, -2.0, 0.0, 3.0e-3], np.float32)
    z = np.zeros(4, np.float32)
    w, m, v = ora.adamw(w0, z, z, z, 0.5, 0.9, 0.95, 1e-8, 0.5, 3)
    assert np.array_equal(w, (w0 - np.float32(0.25) * w0).astype(np.float32))
    assert not m.any() and not v.any()


def test_decay_uses_the_pre_update_weight(ora):
    # w1 = w0 - lr*wd*w0 - lr*u; decaying after the step would give
    # (w0 - lr*u)(1 - lr*wd), which differs by lr^2 wd u.
    w0 = np.array([1.0], np.float32)
    g = np.array([1.0], np.float32)
    z = np.zeros(1, np.float32)
    w, _, _ = ora.adamw(w0, z, z, g, 0.5, 0.9, 0.95, 0.0, 0.5, 1)
    assert w[0] == pytest.approx(1.0 - 0.25 - 0.5, abs=1e-6)
