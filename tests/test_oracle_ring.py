"""Pins of the oracle's collectives against what the pages fix.

* The ring trace for p = 4 printed in CS336 Lecture 7 notes, 4.2.
* Exercise 1 (CS336 Lecture 7 notes, section 11): all-reduce, reduce-scatter
  (rank r keeps chunk r), all-gather of the reduce-scatter, padding for n < p.
* all-reduce = reduce-scatter + all-gather (CS336 Lecture 7 notes 3.4;
  Fudan MLSys ch. 9, 9.3.6) by brute force on small P and n: the per-element
  definition the step uses must equal the literal ring, bit for bit.
* Send volume 2(p-1) messages of n/p per rank (CS336 Lecture 7 notes 4.3;
  the interview guide 2.4) and exercise 2's byte counts.
"""

import numpy as np
import pytest

from conftest import golden
from oracle import accounting


def test_ring_trace_matches_page(ora):
    rows = golden("ring_trace_p4.txt")
    by = {}
    for stage, dev, *vals in rows:
        by.setdefault(stage, {})[int(dev)] = [float(x) for x in vals]
    bufs = np.array([by["init"][d] for d in range(4)], np.float32)
    sent = ora.ring_reduce_scatter_sim(bufs, shift=0)
    for d in range(4):
        assert bufs[d].tolist() == by["after_reduce_scatter_step3"][d]
    assert sent.tolist() == [3, 3, 3, 3]
    ora.ring_all_gather_sim(bufs, shift=0)
    for d in range(4):
        assert bufs[d].tolist() == by["after_all_gather_step3"][d]


def test_owner_schedule_is_the_page_schedule_relabelled(ora):
    # With shift = 0 (the page) device d finishes chunk d+1, summing from
    # device d+1's value round to its own.  With shift = 1 (owner schedule)
    # device c finishes chunk c, summing from device c+1 round to c.  Feeding
    # the page's schedule device d+1's data at device d turns one into the
    # other, bit for bit.
    rng = np.random.default_rng(0)
    for P in (2, 3, 4, 5, 8):
        x = (rng.standard_normal((P, P)) * 10.0 ** rng.integers(-3, 4, (P, P))).astype(np.float32)
        page = np.roll(x, -1, axis=0).copy()  # page[d] = x[d+1]
        own = x.copy()
        ora.ring_reduce_scatter_sim(page, shift=0)
        ora.ring_reduce_scatter_sim(own, shift=1)
        for c in range(P):
            assert page[(c - 1) % P, c].view(np.uint32) == own[c, c].view(np.uint32)


def _bf16_bits(values):
    import torch
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_exercise1(ora):
    rows = golden("exercise1_collectives.txt")
    inputs = np.array([[float(v) for v in r[2:]] for r in rows if r[0] == "input"], np.float32)
    ar = [float(v) for v in next(r for r in rows if r[0] == "all_reduce")[1:]]
    rs = {int(r[1]): [float(r[2])] for r in rows if r[0] == "reduce_scatter"}
    ag = [float(v) for v in next(r for r in rows if r[0] == "all_gather_of_reduce_scatter")[1:]]
    P, n = inputs.shape
    # (b) reduce-scatter by definition: rank r gets chunk r
    shards, flag, _ = ora.reduce_scatter(_bf16_bits(inputs), 0, n, 1.0)
    S = ora.shard_size(n, P)
    for r in range(P):
        assert shards[r * S:(r + 1) * S].tolist() == rs[r]
    assert flag == 0
    # (c) all-gather of (b) = (a)
    rep = ora.all_gather(shards, n, P)
    assert (ora.bf16_to_f32(rep) == np.array(ag, np.float32)).all()
    assert ag == ar
    # the literal ring (owner schedule) gives the same
    bufs = inputs.copy()
    ora.ring_reduce_scatter_sim(bufs, shift=1)
    for r in range(P):
        assert bufs[r, r] == rs[r][0]
    ora.ring_all_gather_sim(bufs, shift=1)
    assert (bufs == np.array(ar, np.float32)).all()


def test_exercise1e_padding(ora):
    # 2 elements per rank cannot be split 4 ways: pad with zeros.
    inputs = np.array([[1, 2], [5, 6], [9, 10], [13, 14]], np.float32)
    P, n = inputs.shape
    S = ora.shard_size(n, P)
    assert S == 1
    shards, _, _ = ora.reduce_scatter(_bf16_bits(inputs), 0, n, 1.0)
    assert shards.tolist() == [28.0, 32.0, 0.0, 0.0]
    rep = ora.all_gather(shards, n, P)
    assert rep.shape == (4, 2)
    assert (ora.bf16_to_f32(rep) == np.array([28, 32], np.float32)).all()


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 7, 8])
def test_definition_equals_literal_ring_bit_for_bit(ora, P):
    rng = np.random.default_rng(P)
    for n in sorted({1, 2, P - 1 if P > 1 else 1, P, P + 1, 7, 17, 64}):
        vals = rng.standard_normal((P, n)).astype(np.float32) * np.float32(10.0) ** rng.integers(-3, 4, (P, n))
        bits = _bf16_bits(vals)
        widened = ora.bf16_to_f32(bits)
        S = ora.shard_size(n, P)
        # literal ring all-reduce on padded fp32 buffers
        bufs = np.zeros((P, P * S), np.float32)
        bufs[:, :n] = widened
        sent_rs = ora.ring_reduce_scatter_sim(bufs, shift=1)
        owned = np.concatenate([bufs[r, r * S:(r + 1) * S] for r in range(P)])
        sent_ag = ora.ring_all_gather_sim(bufs, shift=1)
        # RS followed by AG leaves every rank with the all-reduce
        for r in range(P):
            assert np.array_equal(bufs[r].view(np.uint32), owned.view(np.uint32))
        # the per-element definition gives the identical bits
        shards, _, _ = ora.reduce_scatter(bits, 0, n, 1.0)
        assert np.array_equal(shards.view(np.uint32), owned.view(np.uint32))
        # volume: 2 (P-1) messages of S elements per rank
        assert (sent_rs + sent_ag).tolist() == [2 * (P - 1) * S] * P
        assert int(sent_rs[0] + sent_ag[0]) == accounting.ring_sent_elements_per_rank(n, P)


def test_summation_order_is_observable(ora):
    # The pins above would not notice a wrong order if every order gave the
    # same bits; show that orders differ on these inputs, so they do notice.
    P, n = 8, 4096
    rng = np.random.default_rng(1)
    vals = (rng.standard_normal((P, n)) * 10.0 ** rng.integers(-4, 4, (P, n))).astype(np.float32)
    bits = _bf16_bits(vals)
    shards, _, _ = ora.reduce_scatter(bits, 0, n, 1.0)
    w = ora.bf16_to_f32(bits)
    natural = np.zeros(n, np.float32)
    for q in range(P):
        natural = natural + w[q]
    assert not np.array_equal(shards[:n], natural)


def test_exercise2_volume():
    rows = {r[0]: r[1:] for r in golden("exercise2_volume.txt")}
    p, psi = int(float(rows["p"][0])), float(rows["params"][0])
    ring = accounting.ring_allreduce_bytes_per_rank(psi, p, 2)
    z3 = accounting.zero3_bytes_per_rank(psi, p, 2)
    for key, got in (("ring_bytes_per_gpu", ring), ("ring_seconds_at_50GBps", ring / 50e9),
                     ("zero3_bytes_per_gpu", z3), ("zero3_seconds_at_50GBps", z3 / 50e9)):
        want, tol = float(rows[key][0]), float(rows[key][2])
        assert abs(got - want) <= tol * want + 1e-12, (key, got, want)
    # exactly 1.5x the ring all-reduce (ZeRO-3 moves 3 Psi against 2 Psi)
    assert z3 == pytest.approx(1.5 * ring)
