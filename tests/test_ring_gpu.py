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


@pytest.mark.parametrize("P,n", [(8, 1 << 28), (64, 1 << 26)])
def test_ring_at_the_study_sizes(P, n):
    """The sizes `bench.py --ring-study` times (flat n = 2^28 up to P = 16,
    2^26 at P = 64), against the oracle at sampled indices: every shard edge
    with its neighbours, the ends and random elements."""
    from zero_gradient_reduce_gb300 import workloads

    wl = workloads.Workload(f"flat_{n}_p{P}", P=P, n=n, tensors=workloads._flat(n),
                            fresh_state=True)
    seed = 11
    S = -(-n // P)
    grads = [workloads.fill_grads(torch.empty(n, dtype=torch.bfloat16, device="cuda"), wl, q, 0,
                                  seed) for q in range(P)]
    st = [torch.zeros(P * S, dtype=torch.float32, device="cuda") for _ in range(3)]
    workloads.fill_state(st[0], st[1], st[2], wl, seed)
    reps = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    words = torch.zeros(16, dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(seed)
    pts = {0, n - 1} | {r * S + d for r in range(1, P) for d in range(-8, 8)}
    pts |= set(rng.integers(0, n, 20_000).tolist())
    idx = np.array(sorted(i for i in pts if 0 <= i < n), np.int64)
    idx_dev = torch.from_numpy(idx).to("cuda")
    w, m, v = (x.index_select(0, idx_dev).cpu().numpy().copy() for x in st)
    gs = np.stack([g.index_select(0, idx_dev).view(torch.int16).cpu().numpy().view(np.uint16)
                   for g in grads])
    a, keep = zdp.make_step_args(grads, st[0], st[1], st[2], reps, n=n, scale=wl.scale, t=1,
                                 d_overflow=words[0:4].view(torch.int32),
                                 d_sumsq=words[8:16].view(torch.float64), **HP)
    ws = torch.empty(zdp.zdp_step_ring_workspace_bytes(a), dtype=torch.uint8, device="cuda")
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    zdp.zdp_step_ring(a)
    torch.cuda.synchronize()
    _, rep, flag = oracle.step_sampled(gs, idx, oracle.BF16, w, m, v, n, wl.scale, t=1, **HP)
    label = f"ring P={P} n={n}"
    assert flag == 0 and int(words[0:4].view(torch.int32).item()) == 0
    assert_state_close(st[0].index_select(0, idx_dev).cpu().numpy(), w, label + " master")
    assert_state_close(st[1].index_select(0, idx_dev).cpu().numpy(), m, label + " m")
    assert_state_close(st[2].index_select(0, idx_dev).cpu().numpy(), v, label + " v")
    for q in (0, P // 2, P - 1):
        got = reps[q].index_select(0, idx_dev).view(torch.int16).cpu().numpy().view(np.uint16)
        assert_bf16_close(got, rep, f"{label} replica {q}")
    del grads, st, reps, ws, a, keep
    torch.cuda.empty_cache()
