"""The overflow-checked step in one cooperative launch.

When a range's reduced gradients fit in the registers of one resident wave,
zdp_step with check_overflow makes one cooperative launch with a grid barrier
instead of two passes through the workspace.  The two forms must give the
same bits: the state, the replicas and the flag word.  The sum of squares
agrees to rounding, because its summation order follows the launch shape.
They are compared here across P, sizes, fp32 and bf16 moments and
injected infinities; the environment variable ZDP_COOP=0 forces the two-pass form.
The barrier's wait is bounded; a test makes it run out (it waits for an
arrival that never comes) and checks that the flag word reports it, that
nothing was written, and that the next call works.
"""

import numpy as np
import pytest
import torch

import oracle
from harness import DeviceStep, HP, assert_bits_equal, random_problem

pytestmark = pytest.mark.gpu


def _run(P, n, gbits, w, m, v, rep, bucket=0, coop=True, monkeypatch=None, moments="f32"):
    if monkeypatch is not None:
        monkeypatch.setenv("ZDP_COOP", "1" if coop else "0")
    dev = DeviceStep(P, n, torch.float16, moments=moments)
    dev.load(gbits, w, m, v, rep)
    dev.step(1.0 / (P * 65536.0), 6, check_overflow=True, bucket_elems=bucket)
    torch.cuda.synchronize()
    return dev


def _same(a, b, label):
    for x, y, name in zip(a.state(), b.state(), ("master", "m", "v")):
        assert_bits_equal(x, y, f"{label} {name}")
    assert np.array_equal(a.replica_bits(), b.replica_bits()), f"{label} replicas"
    assert int(a.flag.item()) == int(b.flag.item()), f"{label} flag"
    sa, sb = float(a.sumsq.item()), float(b.sumsq.item())
    if np.isfinite(sb):
        assert abs(sa - sb) <= 1e-12 * abs(sb), (label, sa, sb)
    else:
        assert np.isnan(sa) == np.isnan(sb) and (np.isnan(sb) or sa == sb), (label, sa, sb)


@pytest.mark.parametrize("P", [1, 3, 8, 16, 64])
@pytest.mark.parametrize("n", [1, 9, 4097, 100_003, 1 << 20])
@pytest.mark.parametrize("inject", [False, True])
@pytest.mark.parametrize("moments", ["f32", "bf16"])
def test_single_pass_equals_two_pass(P, n, inject, moments, monkeypatch):
    gbits, w, m, v = random_problem(P, n, P * 7 + n, oracle.FP16)
    if moments == "bf16":
        m, v = oracle.f32_to_bf16(m), oracle.f32_to_bf16(v)
    if inject:
        gbits[P - 1, n // 2] = 0x7C00  # +inf
    rep = np.full((P, n), 0x3F80, np.uint16)
    a = _run(P, n, gbits, w, m, v, rep, coop=True, monkeypatch=monkeypatch, moments=moments)
    b = _run(P, n, gbits, w, m, v, rep, coop=False, monkeypatch=monkeypatch, moments=moments)
    assert int(a.flag.item()) == (1 if inject else 0)
    _same(a, b, f"P={P} n={n} inject={inject}")


@pytest.mark.parametrize("n", [2_000_003, 3_000_001])
def test_single_pass_near_its_capacity_matches_the_oracle(n, monkeypatch):
    # about 2.2-2.5 million elements fit one resident wave: these sizes fall
    # on either side, so one runs the single pass and one the two passes
    P = 8
    gbits, w, m, v = random_problem(P, n, n, oracle.FP16)
    rep = np.zeros((P, n), np.uint16)
    dev = _run(P, n, gbits, w, m, v, rep, monkeypatch=monkeypatch)
    scale = 1.0 / (P * 65536.0)
    flag, ss = oracle.step(gbits, oracle.FP16, w, m, v, rep, n, 0, n, scale, t=6,
                           check_overflow=True, **HP)
    for x, y, name in zip(dev.state(), (w, m, v), ("master", "m", "v")):
        assert_bits_equal(x, y, f"n={n} {name}")
    assert np.array_equal(dev.replica_bits(), rep)
    assert int(dev.flag.item()) == flag
    assert abs(float(dev.sumsq.item()) - ss) <= 1e-9 * ss


def test_barrier_timeout_is_reported_and_writes_nothing(monkeypatch):
    P, n = 8, 50_000
    gbits, w, m, v = random_problem(P, n, 5, oracle.FP16)
    rep = np.full((P, n), 0x1234, np.uint16)
    monkeypatch.setenv("ZDP_TEST_COOP_EXTRA_ARRIVALS", "1")  # one arrival that never comes
    monkeypatch.setenv("ZDP_COOP_TIMEOUT_NS", "2000000")     # 2 ms
    dev = _run(P, n, gbits, w, m, v, rep, monkeypatch=monkeypatch)
    assert int(dev.flag.item()) == 2  # ZDP_FLAG_TIMEOUT, no overflow
    for x, y, name in zip(dev.state(), (w, m, v), ("master", "m", "v")):
        assert_bits_equal(x, y, f"untouched {name}")
    assert np.array_equal(dev.replica_bits(), rep)
    # the context is still usable: the same step without the hook is normal
    monkeypatch.delenv("ZDP_TEST_COOP_EXTRA_ARRIVALS")
    monkeypatch.delenv("ZDP_COOP_TIMEOUT_NS")
    ok = _run(P, n, gbits, w, m, v, rep, monkeypatch=monkeypatch)
    ref = _run(P, n, gbits, w, m, v, rep, coop=False, monkeypatch=monkeypatch)
    assert int(ok.flag.item()) == 0
    _same(ok, ref, "after timeout")


@pytest.mark.parametrize("inject", [False, True])
def test_refused_cooperative_launch_falls_back_to_two_passes(inject, monkeypatch):
    # A cooperative grid far larger than a resident wave (65,536 blocks more)
    # is refused by the runtime before anything runs; the call must then take
    # the two passes and return normally, with the two-pass form's results.
    # (Had the launch been accepted, its barrier could not be met: it would
    # time out and the flag would read 2.)
    P, n = 8, 100_000
    gbits, w, m, v = random_problem(P, n, 17, oracle.FP16)
    if inject:
        gbits[2, 777] = 0xFC00  # -inf
    rep = np.full((P, n), 0x3F80, np.uint16)
    monkeypatch.setenv("ZDP_TEST_COOP_OVERSIZE", "65536")
    a = _run(P, n, gbits, w, m, v, rep, coop=True, monkeypatch=monkeypatch)
    monkeypatch.delenv("ZDP_TEST_COOP_OVERSIZE")
    b = _run(P, n, gbits, w, m, v, rep, coop=False, monkeypatch=monkeypatch)
    assert int(a.flag.item()) == (1 if inject else 0)
    _same(a, b, f"fallback inject={inject}")
