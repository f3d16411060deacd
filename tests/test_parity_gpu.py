"""Parity of the CUDA library with the CPU oracle, element by element, at
sizes the oracle finishes in seconds (several blocks and a ragged tail),
over the edge cases of the step: P from 1 to 64, n from 1 up, shard
boundaries inside a 16-byte vector, misaligned pointers, buckets and
sub-ranges, fp16 gradients with injected infinities and NaNs.

Every call goes through the C ABI (the ctypes binding of libzdp)."""

import numpy as np
import pytest
import torch

import oracle
from harness import (HP, DeviceStep, assert_bf16_close, assert_bits_equal,
                     assert_state_close, bits_of, random_problem)
from zero_gradient_reduce_gb300 import zdp

pytestmark = pytest.mark.gpu

PINF, NINF, NAN16 = 0x7C00, 0xFC00, 0x7E00


def _oracle_step(gbits, w, m, v, rep, n, scale, t, gdt=oracle.BF16, off=0, length=None,
                 check=False):
    length = n - off if length is None else length
    P = gbits.shape[0]
    g = np.ascontiguousarray(gbits[:, off:off + length])
    return oracle.step(g, gdt, w, m, v, rep, n, off, length, scale, t=t,
                       check_overflow=check, **HP)


def _compare_step(dev, w, m, v, rep, flag, sumsq, label):
    gw, gm, gv = dev.state()
    assert_state_close(gw, w, f"{label} master")
    assert_state_close(gm, m, f"{label} m")
    assert_state_close(gv, v, f"{label} v")
    got_rep = dev.replica_bits()
    assert_bf16_close(got_rep, rep[:, :dev.n], f"{label} replicas")
    for q in range(1, dev.P):
        assert_bits_equal(got_rep[q], got_rep[0], f"{label} replica {q} vs 0")
    assert int(dev.flag.item()) == flag, f"{label} flag"
    if sumsq is not None:
        got = float(dev.sumsq.item())
        if np.isfinite(sumsq):
            assert abs(got - sumsq) <= 1e-9 * abs(sumsq) + 1e-300, (label, got, sumsq)
        else:  # an injected inf gives inf, a NaN (or +inf with -inf) gives NaN
            assert got == sumsq or (np.isnan(got) and np.isnan(sumsq)), (label, got, sumsq)


def _full_case(P, n, seed, gdt=oracle.BF16, t=10, misalign=False, **step_kw):
    gbits, w, m, v = random_problem(P, n, seed, gdt)
    rep = np.zeros((P, n), np.uint16)
    dev = DeviceStep(P, n, torch.float16 if gdt == oracle.FP16 else torch.bfloat16,
                     misalign=misalign)
    dev.load(gbits, w, m, v, rep)
    scale = 1.0 / (P * (65536.0 if gdt == oracle.FP16 else 1.0))
    dev.step(scale, t, **step_kw)
    flag, ss = _oracle_step(gbits, w, m, v, rep, n, scale, t, gdt,
                            check=step_kw.get("check_overflow", False))
    return dev, (w, m, v, rep, flag, ss)


# ---------------------------------------------------------------- fused step

def test_tiny_flat_config_full_parity():
    # one flat tensor of 2^20 parameters, P = 4, t = 10
    dev, (w, m, v, rep, flag, ss) = _full_case(4, 1 << 20, seed=1)
    _compare_step(dev, w, m, v, rep, flag, ss, "tiny")


@pytest.mark.parametrize("t", [200, 1000, 1_000_000])
@pytest.mark.parametrize("gdt", [oracle.BF16, oracle.FP16])
def test_fused_step_in_steady_state(t, gdt):
    # From t of a few hundred on, fl(1 - b^t) rounds to exactly 1 (b1 first).
    P, n = 8, 50_003
    dev, (w, m, v, rep, flag, ss) = _full_case(P, n, seed=t % 997, gdt=gdt, t=t)
    _compare_step(dev, w, m, v, rep, flag, ss, f"t={t}")


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8, 16, 17, 64])
def test_fused_step_edge_sizes(P):
    ns = sorted({1, 7, max(P - 1, 1), P, P + 1, 8 * P + 3, 1001, 3 * 8192 + 5})
    for k, n in enumerate(ns):
        dev, (w, m, v, rep, flag, ss) = _full_case(P, n, seed=100 * P + k)
        _compare_step(dev, w, m, v, rep, flag, ss, f"P={P} n={n}")


@pytest.mark.parametrize("P", [3, 8, 64])
def test_shard_boundaries_inside_vectors(P):
    # S not a multiple of 8: the owner changes inside a 16-byte vector
    for n in (P * 8 * 37 + 1, P * 1001, P * 4093 - 2):
        dev, (w, m, v, rep, flag, ss) = _full_case(P, n, seed=n)
        assert dev.S % 8 != 0 or n % P != 0
        _compare_step(dev, w, m, v, rep, flag, ss, f"P={P} n={n}")


@pytest.mark.parametrize("P", [2, 8, 5])
def test_misaligned_pointers_take_the_scalar_path(P):
    dev, (w, m, v, rep, flag, ss) = _full_case(P, 20_003, seed=P, misalign=True)
    _compare_step(dev, w, m, v, rep, flag, ss, f"misaligned P={P}")


def test_first_step_from_fresh_state():
    P, n = 8, 50_000
    gbits, w, m, v = random_problem(P, n, 5, fresh=True)
    rep = np.zeros((P, n), np.uint16)
    dev = DeviceStep(P, n)
    dev.load(gbits, w, m, v, rep)
    dev.step(1.0 / P, 1)
    flag, ss = _oracle_step(gbits, w, m, v, rep, n, 1.0 / P, 1)
    _compare_step(dev, w, m, v, rep, flag, ss, "t=1")


def test_empty_range_is_a_no_op():
    P, n = 4, 1000
    gbits, w, m, v = random_problem(P, n, 6)
    dev = DeviceStep(P, n)
    dev.load(gbits, w, m, v)
    dev.step(0.25, 3, off=500, length=0)
    gw, gm, gv = dev.state()
    assert_bits_equal(gw, w, "master")
    assert int(dev.flag.item()) == 0 and float(dev.sumsq.item()) == 0.0


# ------------------------------------------------------ buckets and sub-ranges

@pytest.mark.parametrize("bucket", [1, 7, 1000, 4099, 1 << 20])
def test_bucket_size_does_not_change_bits(bucket):
    P, n = 8, 123_457
    gbits, w, m, v = random_problem(P, n, 7)
    rep = np.zeros((P, n), np.uint16)
    ref = DeviceStep(P, n)
    ref.load(gbits, w, m, v, rep)
    ref.step(1.0 / P, 4)
    dev = DeviceStep(P, n)
    dev.load(gbits, w, m, v, rep)
    dev.step(1.0 / P, 4, bucket_elems=bucket)
    for a, b, name in zip(dev.state(), ref.state(), ("master", "m", "v")):
        assert_bits_equal(a, b, f"bucket {bucket} {name}")
    assert_bits_equal(dev.replica_bits(), ref.replica_bits(), f"bucket {bucket} replicas")
    flag, ss = _oracle_step(gbits, w, m, v, rep, n, 1.0 / P, 4)
    _compare_step(dev, w, m, v, rep, flag, ss, f"bucket {bucket}")


def test_sub_ranges_compose_to_the_whole_step():
    # streaming the step through calls over [off, off+len) pieces, each with
    # a gradient buffer holding only its piece
    P, n = 5, 100_003
    gbits, w, m, v = random_problem(P, n, 8)
    rep = np.zeros((P, n), np.uint16)
    dev = DeviceStep(P, n)
    dev.load(gbits, w, m, v, rep)
    cuts = [0, 1, 9, 8000, 8003, 40_001, 77_777, n]
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        piece = [torch.empty(hi - lo, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
        for q in range(P):
            piece[q].copy_(dev.grads[q][lo:hi])
        a, keep = zdp.make_step_args(piece, dev.master, dev.m, dev.v, dev.replicas, n=n,
                                     scale=1.0 / P, t=2, off=lo, length=hi - lo,
                                     d_overflow=dev.flag, d_sumsq=dev.sumsq, **HP)
        zdp.zdp_step(a)
    torch.cuda.synchronize()
    flag, ss = _oracle_step(gbits, w, m, v, rep, n, 1.0 / P, 2)
    _compare_step(dev, w, m, v, rep, flag, ss, "sub-ranges")


# ------------------------------------------------------------- unfused calls

@pytest.mark.parametrize("P,n", [(1, 5), (4, 1 << 16), (3, 10_001), (8, 8 * 1000 + 3), (64, 4099)])
def test_reduce_scatter_bit_exact(P, n):
    for gdt, dt in ((oracle.BF16, torch.bfloat16), (oracle.FP16, torch.float16)):
        gbits, _, _, _ = random_problem(P, n, n + gdt, gdt)
        dev = DeviceStep(P, n, dt)
        dev.load(gbits, np.zeros(dev.n_pad), np.zeros(dev.n_pad), np.zeros(dev.n_pad))
        scale = 1.0 / (P * (65536.0 if gdt else 1.0))
        shards = torch.full((dev.n_pad,), float("nan"), dtype=torch.float32, device="cuda")
        zdp.zdp_reduce_scatter(dev.grads, shards, n, P, scale, dev.flag, dev.sumsq)
        want, flag, ss = oracle.reduce_scatter(gbits, gdt, n, scale, want_sumsq=True)
        assert_bits_equal(shards.cpu().numpy(), want, f"RS P={P} n={n} gdt={gdt}")
        assert int(dev.flag.item()) == flag
        assert abs(float(dev.sumsq.item()) - ss) <= 1e-9 * ss


@pytest.mark.parametrize("count", [1, 9, 4096, 100_003])
def test_adamw_shard(count):
    rng = np.random.default_rng(count)
    w = (rng.standard_normal(count) * 0.02).astype(np.float32)
    m = (rng.standard_normal(count) * 1e-4).astype(np.float32)
    v = rng.uniform(0, 1e-6, count).astype(np.float32)
    g = (rng.standard_normal(count) * 1e-3).astype(np.float32)
    d = [torch.from_numpy(x.copy()).cuda() for x in (w, m, v, g)]
    for t in (1, 2, 10):
        zdp.zdp_adamw_shard(d[0], d[1], d[2], d[3], count, t=t, **HP)
        w, m, v = oracle.adamw(w, m, v, g, t=t, **HP)
        torch.cuda.synchronize()
        assert_state_close(d[0].cpu().numpy(), w, "master")
        assert_state_close(d[1].cpu().numpy(), m, "m")
        assert_state_close(d[2].cpu().numpy(), v, "v")


@pytest.mark.parametrize("P,n", [(1, 3), (2, 17), (8, 65_537), (64, 1000)])
def test_all_gather(P, n):
    rng = np.random.default_rng(P * n)
    w = (rng.standard_normal(n) * 10.0 ** rng.integers(-30, 30, n)).astype(np.float32)
    w[:4] = [np.inf, -np.inf, 0.0, -0.0][:min(4, n)] if n >= 4 else w[:4]
    dw = torch.from_numpy(w).cuda()
    reps = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    zdp.zdp_all_gather(dw, reps, n, P)
    want = oracle.all_gather(w, n, P)
    got = np.stack([bits_of(r) for r in reps])
    assert_bf16_close(got, want, "all-gather")


def test_unfused_chain_equals_fused_step():
    P, n = 8, 250_001
    gbits, w, m, v = random_problem(P, n, 9)
    fused = DeviceStep(P, n)
    fused.load(gbits, w, m, v)
    fused.step(1.0 / P, 3)
    chain = DeviceStep(P, n)
    chain.load(gbits, w, m, v)
    shards = torch.empty(chain.n_pad, dtype=torch.float32, device="cuda")
    zdp.zdp_reduce_scatter(chain.grads, shards, n, P, 1.0 / P, chain.flag, chain.sumsq)
    S = chain.S
    for r in range(P):  # each rank updates its own shard
        sl = slice(r * S, (r + 1) * S)
        zdp.zdp_adamw_shard(chain.master[sl], chain.m[sl], chain.v[sl], shards[sl], S, t=3, **HP)
    zdp.zdp_all_gather(chain.master, chain.replicas, n, P)
    torch.cuda.synchronize()
    for a, b, name in zip(chain.state(), fused.state(), ("master", "m", "v")):
        assert_bits_equal(a[:n], b[:n], f"chain {name}")
    assert_bits_equal(chain.replica_bits(), fused.replica_bits(), "chain replicas")
    assert int(chain.flag.item()) == int(fused.flag.item())
    assert float(chain.sumsq.item()) == pytest.approx(float(fused.sumsq.item()), rel=1e-12)


# -------------------------------------------------------- overflow and skip

@pytest.mark.parametrize("P", [2, 8, 64])
def test_fp16_overflow_skip(P):
    n = 33_333
    for case, plan in enumerate([[], [(0, 5, PINF)], [(P - 1, n - 1, NINF)],
                                 [(P // 2, 1234, NAN16)], [(0, 77, PINF), (1, 77, NINF)]]):
        gbits, w, m, v = random_problem(P, n, 1000 * P + case, oracle.FP16)
        for q, i, b in plan:
            gbits[q, i] = b
        rep = np.full((P, n), 0x3F80, np.uint16)
        for check in (True, False):
            dev = DeviceStep(P, n, torch.float16)
            dev.load(gbits, w, m, v, rep)
            scale = 1.0 / (P * 65536.0)
            dev.step(scale, 10, check_overflow=check)
            ww, mm, vv, rr = w.copy(), m.copy(), v.copy(), rep.copy()
            flag, ss = _oracle_step(gbits, ww, mm, vv, rr, n, scale, 10, oracle.FP16, check=check)
            assert flag == (1 if plan else 0)
            _compare_step(dev, ww, mm, vv, rr, flag, ss, f"P={P} case={case} check={check}")


def test_checked_step_without_overflow_matches_single_pass():
    P, n = 8, 200_001
    gbits, w, m, v = random_problem(P, n, 11, oracle.FP16)
    a = DeviceStep(P, n, torch.float16)
    a.load(gbits, w, m, v)
    a.step(1.0 / (P * 65536.0), 5, check_overflow=True, bucket_elems=30_000)
    b = DeviceStep(P, n, torch.float16)
    b.load(gbits, w, m, v)
    b.step(1.0 / (P * 65536.0), 5)
    for x, y, name in zip(a.state(), b.state(), ("master", "m", "v")):
        assert_bits_equal(x, y, f"checked vs single pass {name}")
    assert_bits_equal(a.replica_bits(), b.replica_bits(), "replicas")


@pytest.mark.parametrize("bucket", [1000, 4099, 30_000])
@pytest.mark.parametrize("inject_at", [None, 5, 99_990])
def test_bucketed_checked_step_matches_oracle(bucket, inject_at):
    # Consecutive bucket launches of one call overlap (programmatic dependent
    # launch); the gated update must still see the flag of every bucket's
    # reduce pass, including an infinity in the first or the last bucket.
    P, n = 8, 100_003
    gbits, w, m, v = random_problem(P, n, 21, oracle.FP16)
    if inject_at is not None:
        gbits[3, inject_at] = 0x7C00  # +inf in fp16
    rep = np.full((P, n), 0x3F80, np.uint16)
    dev = DeviceStep(P, n, torch.float16)
    dev.load(gbits, w, m, v, rep)
    scale = 1.0 / (P * 65536.0)
    dev.step(scale, 7, check_overflow=True, bucket_elems=bucket)
    flag, ss = _oracle_step(gbits, w, m, v, rep, n, scale, 7, oracle.FP16, check=True)
    assert flag == (0 if inject_at is None else 1)
    _compare_step(dev, w, m, v, rep, flag, ss, f"bucketed checked {bucket} {inject_at}")


def test_finite_gradients_overflowing_fp32():
    P, n = 2, 4096
    gbits, w, m, v = random_problem(P, n, 12)
    gbits[:, 100] = 0x7F7F  # largest finite bf16 on both ranks: the sum overflows
    rep = np.zeros((P, n), np.uint16)
    dev = DeviceStep(P, n)
    dev.load(gbits, w, m, v, rep)
    dev.step(1.0, 3, check_overflow=True)
    flag, _ = _oracle_step(gbits, w, m, v, rep, n, 1.0, 3, check=True)
    assert flag == 1
    _compare_step(dev, w, m, v, rep, 1, None, "fp32 overflow")


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("moments", ["f32", "bf16"])
def test_sum_of_squares_over_extreme_magnitudes(P, moments):
    # reduced gradients from 1e-30 to 1e30: squares far outside fp32's range
    # must still add up like the oracle's fp64 sum.  The P and moment types
    # cover both forms of the fused kernel's range test (per element, and per
    # vector with its per-element fallback).
    n = 100_003
    rng = np.random.default_rng(13 + P)
    vals = (rng.standard_normal((P, n)) * 10.0 ** rng.uniform(-30, 30, (P, n))).astype(np.float32)
    gbits = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    dev = DeviceStep(P, n, moments=moments)
    zeros = np.zeros(dev.n_pad, np.float32 if moments == "f32" else np.uint16)
    dev.load(gbits, np.zeros(dev.n_pad), zeros, zeros)
    scale = 1.0 / P
    shards = torch.empty(dev.n_pad, dtype=torch.float32, device="cuda")
    zdp.zdp_reduce_scatter(dev.grads, shards, n, P, scale, dev.flag, dev.sumsq)
    want, flag, ss = oracle.reduce_scatter(gbits, oracle.BF16, n, scale, want_sumsq=True)
    assert flag == 0 and int(dev.flag.item()) == 0
    assert np.isfinite(ss) and ss > 1e50
    assert abs(float(dev.sumsq.item()) - ss) <= 1e-9 * ss
    # the same through the fused step
    dev.sumsq.zero_()
    dev.step(scale, 3)
    assert abs(float(dev.sumsq.item()) - ss) <= 1e-9 * ss


# ------------------------------------------------ 12 bytes/param: bf16 moments

@pytest.mark.parametrize("P", [1, 2, 5, 8, 64])
def test_bf16_moments_fused_and_checked(P):
    for n, gdt in ((P * 8 * 61 + 5, oracle.BF16), (40_003, oracle.FP16), (1 << 16, oracle.BF16)):
        gbits, w, m32, v32 = random_problem(P, n, P * 1000 + n, gdt)
        m16, v16 = oracle.f32_to_bf16(m32), oracle.f32_to_bf16(v32)
        scale = 1.0 / (P * (65536.0 if gdt == oracle.FP16 else 1.0))
        for check in (False, True):
            dev = DeviceStep(P, n, torch.float16 if gdt == oracle.FP16 else torch.bfloat16,
                             moments="bf16")
            rep = np.zeros((P, n), np.uint16)
            dev.load(gbits, w, m16, v16, rep)
            dev.step(scale, 4, check_overflow=check)
            ww, mm, vv, rr = w.copy(), m16.copy(), v16.copy(), rep.copy()
            flag, ss = oracle.step(gbits, gdt, ww, mm, vv, rr, n, 0, n, scale, t=4,
                                   check_overflow=check, moments="bf16", **HP)
            label = f"bf16 moments P={P} n={n} check={check}"
            gw, gm, gv = dev.state()
            assert_state_close(gw, ww, label + " master")
            assert_bf16_close(gm, mm, label + " m")
            assert_bf16_close(gv, vv, label + " v")
            assert_bf16_close(dev.replica_bits(), rr, label + " replicas")
            assert int(dev.flag.item()) == flag
            assert abs(float(dev.sumsq.item()) - ss) <= 1e-9 * ss
