"""Pins of the oracle's ZeRO++ pieces (Fudan MLSys ch. 9, 9.4.3: INT8 weights
for the all-gather, block-wise quantized gradients for the reduce-scatter).

The quantizer is pinned to what block absmax quantization must satisfy
(half-step round-trip error, the block maximum at +-127, zero blocks, odd
symmetry, independent blocks, a worked example with a tie), and the ZeRO++ step
to the already-pinned bf16 step: with gradients whose dequantized values are
exact in bf16, it must update master/m/v exactly like the bf16 step and
produce the block quantization of that step's bf16 replicas."""

import numpy as np
import pytest

from harness_cpu import HP, bf16_bits, random_state


def test_round_trip_error_is_at_most_half_a_step(ora):
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(256 * 40 + 77) * 10.0 ** rng.uniform(-8, 3, 256 * 40 + 77)).astype(np.float32)
    q, sc = ora.quantize_blocks(x)
    xr = ora.dequantize_blocks(q, sc)
    step = np.repeat(sc, 256)[:x.size].astype(np.float64)
    assert np.all(np.abs(x.astype(np.float64) - xr) <= step * (0.5 + 1e-5))
    assert np.all(np.abs(q.astype(np.int32)) <= 127)


def test_block_maximum_maps_to_127_and_blocks_are_independent(ora):
    rng = np.random.default_rng(1)
    x = rng.standard_normal(256 * 3 + 10).astype(np.float32)
    x[256:512] *= 1000.0
    q, sc = ora.quantize_blocks(x)
    for b in range(4):
        blk = x[256 * b:256 * (b + 1)]
        k = int(np.argmax(np.abs(blk)))
        assert abs(int(q[256 * b + k])) == 127
        assert sc[b] == np.float32(np.abs(blk).max()) / np.float32(127.0)
    assert sc[1] > 100 * sc[0]


def test_zero_blocks_and_odd_symmetry(ora):
    x = np.zeros(600, np.float32)
    x[300] = -3.0
    x[301] = 1.5
    q, sc = ora.quantize_blocks(x)
    assert sc[0] == 0.0 and not q[:256].any() and sc[2] == 0.0
    qn, scn = ora.quantize_blocks(-x)
    assert np.array_equal(qn, -q) and np.array_equal(scn, sc)


def test_worked_example_with_a_tie(ora):
    x = np.zeros(256, np.float32)
    x[:3] = [1.0, 0.5, -0.25]
    q, sc = ora.quantize_blocks(x)
    # scale = fl(1/127); 0.5/scale rounds to exactly 63.5, a tie -> 64 (even)
    assert sc[0] == np.float32(1.0) / np.float32(127.0)
    assert q[:3].tolist() == [127, 64, -32]


def test_ties_on_an_even_base_round_down(ora):
    # 63.5 -> 64 above is the same under ties-to-even and ties-away; these
    # fp32 inputs divide by fl(1/127) to exactly k + 0.5 with k even, where
    # half-to-even keeps k and half-away would give k + 1 (in magnitude).
    sc = np.float32(1.0) / np.float32(127.0)
    bits = {62.5: 1056700400, 2.5: 1017201285, 0.5: 998310404, 126.5: 1065287164,
            10.5: 1034506917}
    x = np.zeros(256, np.float32)
    x[0] = 1.0
    for k, (tie, b) in enumerate(bits.items()):
        val = np.array([b], np.uint32).view(np.float32)[0]
        assert val / sc == np.float32(tie)  # the premise: an exact tie
        x[1 + 2 * k], x[2 + 2 * k] = val, -val
    q, s = ora.quantize_blocks(x)
    assert s[0] == sc
    want = [127]
    for tie in bits:
        want += [int(tie - 0.5), -int(tie - 0.5)]
    assert q[:len(want)].tolist() == want


def test_zpp_step_equals_bf16_step_when_dequantization_is_exact(ora):
    P, n = 4, 256 * 20 + 37
    rng = np.random.default_rng(2)
    gq = rng.integers(-127, 128, (P, n)).astype(np.int8)
    nb = -(-n // 256)
    gs = np.full((P, nb), 2.0 ** -10, np.float32)  # q * 2^-10 is exact in bf16
    gvals = gq.astype(np.float32) * np.float32(2.0 ** -10)
    gbits = bf16_bits(gvals)
    assert np.array_equal(ora.bf16_to_f32(gbits), gvals)
    w, m, v = random_state(n, rng)
    # the bf16 step
    wa, ma, va = w.copy(), m.copy(), v.copy()
    rep = np.zeros((P, n), np.uint16)
    fa, sa = ora.step(gbits, ora.BF16, wa, ma, va, rep, n, 0, n, 1.0 / P, t=3, **HP)
    # the ZeRO++ step
    wb, mb, vb = w.copy(), m.copy(), v.copy()
    rq = np.zeros((P, n), np.int8)
    rs = np.zeros((P, nb), np.float32)
    fb, sb = ora.step_zpp(gq, gs, wb, mb, vb, rq, rs, n, 0, n, 1.0 / P, t=3, **HP)
    assert np.array_equal(wa.view(np.uint32), wb.view(np.uint32))
    assert np.array_equal(ma.view(np.uint32), mb.view(np.uint32))
    assert np.array_equal(va.view(np.uint32), vb.view(np.uint32))
    assert (fa, sa) == (fb, sb)
    want_q, want_s = ora.quantize_blocks(ora.bf16_to_f32(rep[0]))
    for q in range(P):
        assert np.array_equal(rq[q], want_q) and np.array_equal(rs[q], want_s)


def test_zpp_step_on_a_block_range_equals_the_whole(ora):
    P, n = 3, 256 * 12 + 5
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((P, n)) * 1e-3).astype(np.float32)
    qs = [ora.quantize_blocks(x[r]) for r in range(P)]
    gq = np.stack([a for a, _ in qs])
    gs = np.stack([b for _, b in qs])
    w, m, v = random_state(n, rng)
    nb = gs.shape[1]
    wa, ma, va = w.copy(), m.copy(), v.copy()
    rqa, rsa = np.zeros((P, n), np.int8), np.zeros((P, nb), np.float32)
    ora.step_zpp(gq, gs, wa, ma, va, rqa, rsa, n, 0, n, 1.0 / P, t=5, **HP)
    # blocks 4..8 alone, with buffers holding only that range
    lo, hi = 256 * 4, 256 * 9
    wb, mb, vb = w[lo:hi].copy(), m[lo:hi].copy(), v[lo:hi].copy()
    rqb, rsb = np.zeros((P, hi - lo), np.int8), np.zeros((P, 5), np.float32)
    ora.step_zpp(np.ascontiguousarray(gq[:, lo:hi]), np.ascontiguousarray(gs[:, 4:9]), wb, mb,
                 vb, rqb, rsb, n, lo, hi - lo, 1.0 / P, t=5, base=lo, **HP)
    assert np.array_equal(wb, wa[lo:hi]) and np.array_equal(rqb, rqa[:, lo:hi])
    assert np.array_equal(rsb, rsa[:, 4:9])


def test_non_finite_blocks_dequantize_to_non_finite_values(ora):
    # The page leaves non-finite inputs open; the reading: a NaN makes the
    # block's maximum (so its scale) NaN, an infinity makes it infinite, and a
    # NaN quotient takes the clamp's lower end, -127.  Every element of such a
    # block then dequantizes to a non-finite value (q * NaN, 0 * inf, -127 *
    # inf), while the other blocks quantize as if nothing happened.
    rng = np.random.default_rng(9)
    x = rng.standard_normal(256 * 4).astype(np.float32)
    clean_q, clean_sc = ora.quantize_blocks(x)
    x[256 + 17] = np.nan
    x[512 + 3] = np.inf
    x[768 + 200] = -np.inf
    q, sc = ora.quantize_blocks(x)
    assert np.isnan(sc[1]) and sc[2] == np.inf and sc[3] == np.inf
    assert (q[256:512] == -127).all()
    for b, k in ((2, 3), (3, 200)):
        blk = q[256 * b:256 * (b + 1)]
        assert blk[k] == -127 and not np.delete(blk, k).any()
    assert np.array_equal(q[:256], clean_q[:256]) and sc[0] == clean_sc[0]
    xr = ora.dequantize_blocks(q, sc)
    assert not np.isfinite(xr[256:]).any() and np.isfinite(xr[:256]).all()


@pytest.mark.parametrize("bad", [np.nan, np.inf])
def test_zpp_step_reports_a_non_finite_gradient(ora, bad):
    # One rank's gradient holds a NaN or an infinity before quantization: the
    # block's dequantized values, hence the reduced gradients there, are not
    # finite and the step's overflow flag is raised; other blocks are unharmed.
    P, n = 4, 256 * 8
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((P, n)) * 1e-3).astype(np.float32)
    x[2, 256 * 5 + 9] = bad
    gq = np.empty((P, n), np.int8)
    gs = np.empty((P, n // 256), np.float32)
    for q in range(P):
        gq[q], gs[q] = ora.quantize_blocks(x[q])
    w, m, v = random_state(n, rng)
    rq = np.zeros((P, n), np.int8)
    rs = np.zeros((P, n // 256), np.float32)
    flag, _ = ora.step_zpp(gq, gs, w, m, v, rq, rs, n, 0, n, 1.0 / P, t=3, **HP)
    assert flag == 1
    assert not np.isfinite(w[256 * 5:256 * 6]).any()
    assert np.isfinite(w[:256 * 5]).all() and np.isfinite(w[256 * 6:]).all()
