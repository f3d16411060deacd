"""Pins of the oracle's overflow flag and skip (a reading: the pages have no
loss-scale overflow check; the flag is "some reduced gradient is not
finite", and a checked step then writes nothing)."""

import numpy as np

PINF, NINF, NAN16 = 0x7C00, 0xFC00, 0x7E00


def _setup(P=4, n=64, seed=0):
    rng = np.random.default_rng(seed)
    g = (rng.standard_normal((P, n)) * 64).astype(np.float16).view(np.uint16).copy()
    w = rng.standard_normal(n).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = rng.uniform(0, 1e-6, n).astype(np.float32)
    rep = np.full((P, n), 0x1234, np.uint16)
    return g, w, m, v, rep


def _run(ora, g, w, m, v, rep, check):
    P, n = g.shape
    return ora.step(g, 1, w, m, v, rep, n, 0, n, 1.0 / (P * 65536.0), 1e-4, 0.9, 0.95, 1e-8,
                    0.1, 10, check_overflow=check)


def test_clean_step_has_no_flag(ora):
    g, w, m, v, rep = _setup()
    flag, _ = _run(ora, g, w.copy(), m.copy(), v.copy(), rep.copy(), True)
    assert flag == 0


def test_injected_values_raise_the_flag_and_skip(ora):
    for q, i, bits in [(0, 3, PINF), (2, 10, NINF), (3, 63, NAN16)]:
        g, w, m, v, rep = _setup()
        g[q, i] = bits
        w1, m1, v1, r1 = w.copy(), m.copy(), v.copy(), rep.copy()
        flag, _ = _run(ora, g, w1, m1, v1, r1, True)
        assert flag == 1
        assert np.array_equal(w1, w) and np.array_equal(m1, m) and np.array_equal(v1, v)
        assert np.array_equal(r1, rep)


def test_opposite_infinities_sum_to_nan(ora):
    g, w, m, v, rep = _setup()
    g[0, 5], g[1, 5] = PINF, NINF
    shards, flag, _ = ora.reduce_scatter(g, 1, g.shape[1], 1.0)
    assert flag == 1 and np.isnan(shards[5])


def test_finite_inputs_overflowing_fp32_raise_the_flag(ora):
    P, n = 2, 8
    g = np.zeros((P, n), np.uint16)
    g[:, 2] = 0x7F7F  # largest finite bf16, ~3.39e38; two of them overflow fp32
    shards, flag, _ = ora.reduce_scatter(g, 0, n, 0.5)
    assert flag == 1 and np.isinf(shards[2])


def test_unchecked_step_writes_despite_the_flag(ora):
    g, w, m, v, rep = _setup()
    g[1, 7] = PINF
    w1, m1, v1, r1 = w.copy(), m.copy(), v.copy(), rep.copy()
    flag, _ = _run(ora, g, w1, m1, v1, r1, False)
    assert flag == 1
    assert np.isnan(w1[7]) or np.isinf(w1[7])
    assert not np.array_equal(r1, rep)
