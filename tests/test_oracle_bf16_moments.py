"""Pins of the oracle's bf16-moment step against its pinned fp32 path.

With moments stored in bf16 (CS336 Lecture 7 notes, 8.4), one step must equal
the fp32-moment step run on the widened bf16 moments -- the same master weight
and replicas -- with the new moments rounded to nearest even on the way out.
Both the fp32 step and the rounding are pinned elsewhere, so a wrong widening,
a rounding in the wrong place or an update computed from the rounded moments
fails here."""

import numpy as np

from harness_cpu import HP, bf16_bits, random_state


def test_bf16_moments_step_equals_rounded_fp32_step(ora):
    P, n = 4, 50_000
    rng = np.random.default_rng(3)
    g = bf16_bits(rng.standard_normal((P, n)) * 1e-3)
    w, m32, v32 = random_state(n, rng)
    m16, v16 = ora.f32_to_bf16(m32), ora.f32_to_bf16(v32)
    # fp32 path on the widened moments
    wa, ma, va = w.copy(), ora.bf16_to_f32(m16), ora.bf16_to_f32(v16)
    rep_a = np.zeros((P, n), np.uint16)
    ora.step(g, ora.BF16, wa, ma, va, rep_a, n, 0, n, 1.0 / P, t=7, **HP)
    # bf16-moment path
    wb, mb, vb = w.copy(), m16.copy(), v16.copy()
    rep_b = np.zeros((P, n), np.uint16)
    ora.step(g, ora.BF16, wb, mb, vb, rep_b, n, 0, n, 1.0 / P, t=7, moments="bf16", **HP)
    assert np.array_equal(wa.view(np.uint32), wb.view(np.uint32))
    assert np.array_equal(rep_a, rep_b)
    assert np.array_equal(mb, ora.f32_to_bf16(ma))
    assert np.array_equal(vb, ora.f32_to_bf16(va))


def test_sampled_step_with_bf16_moments(ora):
    P, n = 8, 10_000
    rng = np.random.default_rng(4)
    g = bf16_bits(rng.standard_normal((P, n)) * 1e-3)
    w, m32, v32 = random_state(n, rng)
    m16, v16 = ora.f32_to_bf16(m32), ora.f32_to_bf16(v32)
    wf, mf, vf = w.copy(), m16.copy(), v16.copy()
    rep = np.zeros((P, n), np.uint16)
    ora.step(g, ora.BF16, wf, mf, vf, rep, n, 0, n, 1.0 / P, t=2, moments="bf16", **HP)
    idx = np.sort(rng.choice(n, 500, replace=False)).astype(np.int64)
    ws, ms, vs = w[idx].copy(), m16[idx].copy(), v16[idx].copy()
    _, rs, _ = ora.step_sampled(np.ascontiguousarray(g[:, idx]), idx, ora.BF16, ws, ms, vs, n,
                                1.0 / P, t=2, moments="bf16", **HP)
    assert np.array_equal(ws, wf[idx]) and np.array_equal(ms, mf[idx])
    assert np.array_equal(vs, vf[idx]) and np.array_equal(rs, rep[0, idx])
