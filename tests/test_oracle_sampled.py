"""Pins of the oracle's sampled step against its whole-range step.

The parity tests at full model size check the library only at sampled global
indices, with ``oracle.step_sampled`` computing the expected values one by one.
That function must therefore give, at every sampled index, exactly what the
whole-range step gives there.  The whole-range step and the reduce-scatter are
pinned elsewhere (the ring trace and exercises of CS336 Lecture 7 notes 4.2
and 11, the Adam closed forms of Fudan MLSys ch. 9, 9.2.2, the overflow
cases), so these tests carry those pins over to the sampled form, for each
branch it has: fp32 and bf16 moments, bf16 and fp16 gradients, and the skip
of an overflowed step.  The samples are chosen so that the owner of a sampled
element differs from the owner of its position in the sample, which catches an
owner computed from the wrong index.
"""

import numpy as np
import pytest

from harness_cpu import HP, bf16_bits, random_state


def _fp16_bits(x):
    return np.ascontiguousarray(np.asarray(x, np.float32).astype(np.float16)).view(np.uint16)


def _sample(n, P, rng, k=600):
    """Sorted global indices: every shard's first and last element, the
    model's last element, and random ones."""
    S = -(-n // P)
    edges = {min(n - 1, r * S + d) for r in range(P) for d in (0, S - 1)} | {n - 1}
    rest = rng.choice(n, k, replace=False)
    return np.array(sorted(edges | set(int(i) for i in rest)), np.int64)


def _problem(P, n, gdt, moments, seed):
    import oracle

    rng = np.random.default_rng(seed)
    # magnitudes spread over many binades, so that the fp32 ring sum depends on
    # where the ring starts (a sum of a few bf16 values of similar size is
    # exact in any order, and would hide a wrong owner)
    x = rng.standard_normal((P, n))
    if gdt == oracle.FP16:
        x *= 10.0 ** rng.uniform(-9.0, -0.7, (P, n))
        g, scale = _fp16_bits(x * 65536.0), 1.0 / (P * 65536.0)
    else:
        x *= 10.0 ** rng.uniform(-7.0, 1.0, (P, n))
        g, scale = bf16_bits(x), 1.0 / P
    w, m, v = random_state(n, rng)
    if moments == "bf16":
        m, v = oracle.f32_to_bf16(m), oracle.f32_to_bf16(v)
    return rng, g, scale, w, m, v


@pytest.mark.parametrize("gdt_name", ["bf16", "fp16"])
@pytest.mark.parametrize("moments", ["f32", "bf16"])
@pytest.mark.parametrize("P,n", [(8, 10_007), (3, 4_099), (5, 2_001)])
def test_sampled_step_equals_the_whole_step(ora, gdt_name, moments, P, n):
    gdt = ora.FP16 if gdt_name == "fp16" else ora.BF16
    rng, g, scale, w, m, v = _problem(P, n, gdt, moments, seed=P * 1000 + n)
    wf, mf, vf = w.copy(), m.copy(), v.copy()
    rep = np.zeros((P, n), np.uint16)
    flag, _ = ora.step(g, gdt, wf, mf, vf, rep, n, 0, n, scale, t=3, moments=moments, **HP)
    shards, rs_flag, _ = ora.reduce_scatter(g, gdt, n, scale)
    idx = _sample(n, P, rng)
    ws, ms, vs = w[idx].copy(), m[idx].copy(), v[idx].copy()
    gout, rs, sflag = ora.step_sampled(np.ascontiguousarray(g[:, idx]), idx, gdt, ws, ms, vs, n,
                                       scale, t=3, moments=moments, **HP)
    assert np.array_equal(gout.view(np.uint32), shards[idx].view(np.uint32))
    assert np.array_equal(ws.view(np.uint32), wf[idx].view(np.uint32))
    assert np.array_equal(ms, mf[idx]) and np.array_equal(vs, vf[idx])
    for q in range(P):
        assert np.array_equal(rs, rep[q, idx])
    assert sflag == flag == rs_flag == 0
    # the inputs do make the start of the ring matter at the sampled indices
    wrong, _, _ = ora.step_sampled(np.ascontiguousarray(np.roll(g[:, idx], 1, axis=0)), idx,
                                   gdt, w[idx].copy(), m[idx].copy(), v[idx].copy(), n, scale,
                                   t=3, moments=moments, **HP)
    assert not np.array_equal(wrong.view(np.uint32), gout.view(np.uint32))


@pytest.mark.parametrize("moments", ["f32", "bf16"])
def test_sampled_skip_equals_the_skipped_whole_step(ora, moments):
    # fp16 gradients with an infinity in one rank: the checked whole step
    # writes nothing, so its replicas keep what the previous step left there
    # (here the bf16 of the current master), and the sampled step with skip
    # must leave the state as it was and report those same replicas.
    P, n = 8, 10_007
    rng, g, scale, w, m, v = _problem(P, n, ora.FP16, moments, seed=77)
    bad = 3 * (-(-n // P)) + 11   # an element of rank 3's shard
    g[5, bad] = 0x7C00            # +inf from rank 5
    wf, mf, vf = w.copy(), m.copy(), v.copy()
    before = ora.f32_to_bf16(w)
    rep = np.tile(before, (P, 1))
    flag, _ = ora.step(g, ora.FP16, wf, mf, vf, rep, n, 0, n, scale, t=3, check_overflow=True,
                       moments=moments, **HP)
    assert flag == 1
    assert np.array_equal(wf.view(np.uint32), w.view(np.uint32))
    idx = np.unique(np.concatenate([_sample(n, P, rng), [bad]])).astype(np.int64)
    ws, ms, vs = w[idx].copy(), m[idx].copy(), v[idx].copy()
    gout, rs, sflag = ora.step_sampled(np.ascontiguousarray(g[:, idx]), idx, ora.FP16, ws, ms,
                                       vs, n, scale, t=3, skip=True, moments=moments, **HP)
    assert sflag == 1
    assert np.isinf(gout[np.searchsorted(idx, bad)])
    assert np.array_equal(ws.view(np.uint32), w[idx].view(np.uint32))
    assert np.array_equal(ms, m[idx]) and np.array_equal(vs, v[idx])
    assert np.array_equal(rs, before[idx]) and np.array_equal(rs, rep[0, idx])
