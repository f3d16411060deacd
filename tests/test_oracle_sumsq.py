"""Closed-form pins of the oracle's overflow word and sum of squares.

The pages use the global gradient norm to clip gradients.  The step returns
the sum of squares of the reduced gradient; the norm is its square root.
Here every rank holds the same value c_i = k_i / 64 (k_i an integer,
|k_i| <= 255, exact in bf16 and in int8 * 2^-6), P is a power of two and the
scale is 1/P.  Each fp32 partial sum j * c_i is then exact, and so is the
multiply by 1/P.  The reduced gradient is therefore c_i exactly, and the sum
of squares is the integer sum of k_i^2 divided by 4096, exact in fp64.  The
expected value comes from Python integers alone, not from the oracle's
arithmetic.
"""

import numpy as np
import pytest

from harness_cpu import HP, bf16_bits


def _problem(P, n, seed):
    rng = np.random.default_rng(seed)
    k = rng.integers(-255, 256, n)
    c = k.astype(np.float32) / np.float32(64.0)
    want = sum(int(x) * int(x) for x in k) / 4096.0
    return k, c, want


@pytest.mark.parametrize("P,n", [(1, 1000), (4, 4097), (8, 20_000), (16, 3 * 256 + 5)])
def test_step_sum_of_squares_closed_form(ora, P, n):
    k, c, want = _problem(P, n, P)
    g = np.repeat(bf16_bits(c)[None, :], P, axis=0)
    S = ora.shard_size(n, P)
    w = np.zeros(P * S, np.float32)
    m = np.zeros(P * S, np.float32)
    v = np.zeros(P * S, np.float32)
    rep = np.zeros((P, n), np.uint16)
    flag, ss = ora.step(g, ora.BF16, w, m, v, rep, n, 0, n, 1.0 / P, t=1, **HP)
    assert flag == 0 and ss == want
    shards, flag2, ss2 = ora.reduce_scatter(g, ora.BF16, n, 1.0 / P, want_sumsq=True)
    assert flag2 == 0 and ss2 == want
    assert np.array_equal(shards[:n], c)


def test_squares_are_taken_in_fp64(ora):
    # Ranks 0..2 hold c, c * 2^-8 and c * 2^-16, rank 3 holds 0, with
    # c = k / 64 and |k| <= 15.  The three copies of k's bits do not overlap,
    # so every partial ring sum is exact in fp32 (20 significant bits), but
    # its square (40 bits) is not: an fp32 square would round.  The fp64
    # squares and their running sum stay exact (below 2^53 units of 2^-48).
    P, n = 4, 4097
    rng = np.random.default_rng(11)
    k = rng.integers(-15, 16, n)
    c = k.astype(np.float32) / np.float32(64.0)
    rows = np.stack([c, c * np.float32(2.0 ** -8), c * np.float32(2.0 ** -16), 0 * c])
    g = bf16_bits(rows)
    assert np.array_equal(ora.bf16_to_f32(g), rows)
    # g_i = (k_i / 64) * (65793 / 65536) / 4 = k_i * 65793 * 2^-24
    want = sum((int(x) * 65793) ** 2 for x in k) * 2.0 ** -48
    S = ora.shard_size(n, P)
    w, m, v = (np.zeros(P * S, np.float32) for _ in range(3))
    rep = np.zeros((P, n), np.uint16)
    flag, ss = ora.step(g, ora.BF16, w, m, v, rep, n, 0, n, 1.0 / P, t=1, **HP)
    assert flag == 0 and ss == want
    _, _, ss2 = ora.reduce_scatter(g, ora.BF16, n, 1.0 / P, want_sumsq=True)
    assert ss2 == want


@pytest.mark.parametrize("P,n", [(2, 256 * 9 + 17), (8, 256 * 40)])
def test_zpp_sum_of_squares_closed_form(ora, P, n):
    # Every rank holds int8 codes k_i with the block scale s = 3049 * 2^-20
    # (12 significant bits): each partial sum j * k_i * s (j <= 8) is exact in
    # fp32, the squares (38 bits) are exact only in fp64.
    rng = np.random.default_rng(100 + P)
    k = rng.integers(-127, 128, n)
    want = sum(int(x) * int(x) for x in k) * 3049 ** 2 * 2.0 ** -40
    gq = np.repeat(k.astype(np.int8)[None, :], P, axis=0)
    nb = -(-n // 256)
    gs = np.full((P, nb), 3049 * 2.0 ** -20, np.float32)
    S = ora.shard_size(n, P)
    w = np.zeros(P * S, np.float32)
    m = np.zeros(P * S, np.float32)
    v = np.zeros(P * S, np.float32)
    rq = np.zeros((P, n), np.int8)
    rs = np.zeros((P, nb), np.float32)
    flag, ss = ora.step_zpp(gq, gs, w, m, v, rq, rs, n, 0, n, 1.0 / P, t=1, **HP)
    assert flag == 0 and ss == want


def test_sum_of_squares_adds_over_calls(ora):
    # Two half-range calls add into the caller's sum; the halves' closed forms add up.
    P, n = 4, 2048
    k, c, want = _problem(P, n, 5)
    g = np.repeat(bf16_bits(c)[None, :], P, axis=0)
    w = np.zeros(n, np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    rep = np.zeros((P, n), np.uint16)
    total = 0.0
    for lo, hi in ((0, 1000), (1000, n)):
        _, s = ora.step(np.ascontiguousarray(g[:, lo:hi]), ora.BF16, w[lo:], m[lo:], v[lo:],
                        np.ascontiguousarray(rep[:, lo:]), n, lo, hi - lo, 1.0 / P, t=1,
                        base=lo, **HP)
        assert s == sum(int(x) * int(x) for x in k[lo:hi]) / 4096.0
        total += s
    assert total == want
