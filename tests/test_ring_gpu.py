"""zdp_step_ring: the step run as the literal ring schedule (one launch per
ring step, fp32 partial sums passed between the ranks' message buffers).
Its additions happen in the fused kernel's order, so it must give the
oracle's bits, and zdp_step's, exactly."""

import numpy as np
import pytest
import torch

import oracle
from harness import (HP, DeviceStep, assert_bf16_close, assert_bits_equal, assert_state_close,
                     random_problem)
from zero_gradient_reduce_gb300 import zdp

pytestmark = pytest.mark.gpu


def _ring(dev, scale, t, gdt_fp16=False):
    a, keep = dev.args(scale, t)
    ws = torch.empty(zdp.zdp_step_ring_workspace_bytes(a), dtype=torch.uint8, device="cuda")
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    zdp.zdp_step_ring(a)
    torch.cuda.synchronize()
    return keep, ws


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16])
def test_ring_matches_the_oracle(P):
    for n in sorted({1, P + 1, 8 * P * 5, 8 * P * 5 + 3, 10_007, 65_536}):
        gbits, w, m, v = random_problem(P, n, 7 * P + n)
        rep = np.zeros((P, n), np.uint16)
        dev = DeviceStep(P, n)
        dev.load(gbits, w, m, v, rep)
        _ring(dev, 1.0 / P, 6)
        flag, ss = oracle.step(gbits, oracle.BF16, w, m, v, rep, n, 0, n, 1.0 / P, t=6, **HP)
        gw, gm, gv = dev.state()
        label = f"ring P={P} n={n}"
        assert_state_close(gw[:n], w[:n], label + " master")
        assert_state_close(gm[:n], m[:n], label + " m")
        assert_state_close(gv[:n], v[:n], label + " v")
        reps = dev.replica_bits()
        for q in range(P):
            assert_bf16_close(reps[q], rep[q], f"{label} replica {q}")
        assert int(dev.flag.item()) == flag
        assert abs(float(dev.sumsq.item()) - ss) <= 1e-9 * ss


@pytest.mark.parametrize("P,n,fp16", [(8, 1_000_000, False), (5, 333_337, True), (64, 65_536, False)])
def test_ring_is_bit_identical_to_the_fused_step(P, n, fp16):
    gdt = oracle.FP16 if fp16 else oracle.BF16
    gbits, w, m, v = random_problem(P, n, P * n, gdt)
    dt = torch.float16 if fp16 else torch.bfloat16
    scale = 1.0 / (P * (65536.0 if fp16 else 1.0))
    fused, ring = DeviceStep(P, n, dt), DeviceStep(P, n, dt)
    for d in (fused, ring):
        d.load(gbits, w, m, v)
    fused.step(scale, 3)
    _ring(ring, scale, 3)
    for a, b, name in zip(ring.state(), fused.state(), ("master", "m", "v")):
        assert_bits_equal(a[:n], b[:n], f"ring vs fused {name}")
    assert_bits_equal(ring.replica_bits(), fused.replica_bits(), "ring vs fused replicas")
    assert int(ring.flag.item()) == int(fused.flag.item())
    assert float(ring.sumsq.item()) == pytest.approx(float(fused.sumsq.item()), rel=1e-12)
