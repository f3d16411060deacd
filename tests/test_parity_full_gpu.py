"""Parity at the workloads' full sizes, in the launch configurations the
benchmark and a training loop use, on sampled outputs the oracle computes one
by one.

The step is elementwise once the owner of an element is known, so the oracle
can follow any set of elements through any number of steps on its own: it
takes the gradient values at the sampled global indices (copied from the
device inputs), its own copy of the state at those indices, and produces the
reduced gradient, the new state and the bf16 replica value of each.  Samples
cover every shard boundary, bucket boundary and tensor boundary (with their
neighbours), the ends of the range, every injected infinity or NaN, and
random elements.

The overflow flag is checked against a property that holds at any size: the
workloads' gradients are bounded (|bf16| < 1, |fp16| <= 65504, at most 64
ranks), so no sum of them overflows fp32, and the flag is raised exactly when
an injected infinity or NaN reaches a reduced gradient; all injected
positions are in the sample.
"""

import gc

import numpy as np
import pytest
import torch

import oracle
from harness import (HP, SampledProducer, assert_bf16_close, assert_bits_equal,
                     assert_state_close, bits_of)
from zero_gradient_reduce_gb300 import streaming, workloads, zdp

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def sample_indices(n, S, P, seed, extra=(), k_random=20_000, around=16):
    pts = [0, n - 1]
    pts += [r * S for r in range(1, P) if r * S < n]
    pts += list(extra)
    out = set()
    for b in pts:
        for d in range(-around, around + 1):
            if 0 <= b + d < n:
                out.add(int(b + d))
    rng = np.random.default_rng(seed)
    out.update(int(x) for x in rng.integers(0, n, min(k_random, n)))
    return np.array(sorted(out), np.int64)


def gather_bits(t, idx_dev):
    return bits_of(t.index_select(0, idx_dev))


def gather_f32(t, idx_dev):
    return t.index_select(0, idx_dev).cpu().numpy()


class Problem:
    """Full-size device buffers of one workload."""

    def __init__(self, wl, seed, grads=True, moments="f32"):
        self.wl, self.P, self.n = wl, wl.P, wl.n
        self.S = -(-wl.n // wl.P)
        self.moments = moments
        gdt = torch.float16 if wl.grad_dtype == "fp16" else torch.bfloat16
        self.grads = ([torch.empty(wl.n, dtype=gdt, device=DEV) for _ in range(wl.P)]
                      if grads else None)
        self.state = torch.empty(3, self.P * self.S, dtype=torch.float32, device=DEV)
        workloads.fill_state(self.state[0], self.state[1], self.state[2], wl, seed)
        if moments == "bf16":  # the same moments, held in bf16
            self.mv16 = self.state[1:].to(torch.bfloat16)
            self.state = self.state[:1].clone()
        self.replicas = [torch.full((wl.n,), 0.5, dtype=torch.bfloat16, device=DEV)
                         for _ in range(wl.P)]
        self.words = torch.zeros(16, dtype=torch.uint8, device=DEV)
        self.flag = self.words[0:4].view(torch.int32)
        self.sumsq = self.words[8:16].view(torch.float64)

    def buffers(self):
        if self.moments == "f32":
            return self.state[0], self.state[1], self.state[2]
        return self.state[0], self.mv16[0], self.mv16[1]

    def oracle_state(self, idx_dev):
        if self.moments == "f32":
            return [gather_f32(self.state[k], idx_dev).copy() for k in range(3)]
        return [gather_f32(self.state[0], idx_dev).copy(), gather_bits(self.mv16[0], idx_dev),
                gather_bits(self.mv16[1], idx_dev)]

    def check(self, idx, idx_dev, ora_w, ora_m, ora_v, ora_rep, label):
        assert_state_close(gather_f32(self.state[0], idx_dev), ora_w, f"{label} master")
        if self.moments == "f32":
            for k, (name, want) in enumerate((("m", ora_m), ("v", ora_v)), start=1):
                assert_state_close(gather_f32(self.state[k], idx_dev), want, f"{label} {name}")
        else:
            assert_bf16_close(gather_bits(self.mv16[0], idx_dev), ora_m, f"{label} m")
            assert_bf16_close(gather_bits(self.mv16[1], idx_dev), ora_v, f"{label} v")
        reps = np.stack([gather_bits(r, idx_dev) for r in self.replicas])
        for q in range(self.P):
            assert_bf16_close(reps[q], ora_rep, f"{label} replica {q}")


def test_gpt2_small_bucketed_ten_steps():
    wl = workloads.gpt2_small()
    seed = 2
    pb = Problem(wl, seed)
    B = wl.bucket_elems
    tensor_edges = [t.offset for t in wl.tensors]
    idx = sample_indices(pb.n, pb.S, pb.P, seed, extra=list(range(0, pb.n, B)) + tensor_edges,
                         k_random=30_000, around=8)
    idx_dev = torch.from_numpy(idx).to(DEV)
    w, m, v = pb.oracle_state(idx_dev)
    args, keep = zdp.make_step_args(pb.grads, pb.state[0], pb.state[1], pb.state[2],
                                    pb.replicas, n=pb.n, scale=wl.scale, t=1, bucket_elems=B,
                                    d_overflow=pb.flag, d_sumsq=pb.sumsq, **HP)
    for t in range(1, wl.steps + 1):
        for q in range(pb.P):
            workloads.fill_grads(pb.grads[q], wl, q, t, seed)
        gs = np.stack([gather_bits(g, idx_dev) for g in pb.grads])
        pb.words.zero_()
        args.t = t
        zdp.zdp_step(args)
        torch.cuda.synchronize()
        gout, rep, flag = oracle.step_sampled(gs, idx, oracle.BF16, w, m, v, pb.n, wl.scale,
                                              t=t, **HP)
        assert flag == 0 and int(pb.flag.item()) == 0
        pb.check(idx, idx_dev, w, m, v, rep, f"gpt2 t={t}")
    del pb, args, keep
    _free()


@pytest.mark.parametrize("moments", ["f32", "bf16"])
def test_gpt_1p3b_bench_configuration(moments):
    # one fused zdp_step over the whole model per step, flag and sum of
    # squares on, no buckets: the call the benchmark times (with fp32 or
    # bf16 moments)
    wl = workloads.gpt_1p3b()
    seed = 3
    pb = Problem(wl, seed, moments=moments)
    idx = sample_indices(pb.n, pb.S, pb.P, seed, extra=[t.offset for t in wl.tensors],
                         k_random=50_000, around=8)
    idx_dev = torch.from_numpy(idx).to(DEV)
    w, m, v = pb.oracle_state(idx_dev)
    args, keep = zdp.make_step_args(pb.grads, *pb.buffers(), pb.replicas, n=pb.n,
                                    scale=wl.scale, t=1, d_overflow=pb.flag, d_sumsq=pb.sumsq,
                                    moments=moments, **HP)
    for t in range(1, wl.steps + 1):
        for q in range(pb.P):
            workloads.fill_grads(pb.grads[q], wl, q, t, seed)
        gs = np.stack([gather_bits(g, idx_dev) for g in pb.grads])
        pb.words.zero_()
        args.t = t
        zdp.zdp_step(args)
        torch.cuda.synchronize()
        gout, rep, flag = oracle.step_sampled(gs, idx, oracle.BF16, w, m, v, pb.n, wl.scale,
                                              t=t, moments=moments, **HP)
        assert flag == 0 and int(pb.flag.item()) == 0
        assert float(pb.sumsq.item()) > 0.0
        pb.check(idx, idx_dev, w, m, v, rep, f"1.3B {moments} moments t={t}")
    # the reduced gradients of the last step, bit for bit
    shards = torch.empty(pb.P * pb.S, dtype=torch.float32, device=DEV)
    zdp.zdp_reduce_scatter(pb.grads, shards, pb.n, pb.P, wl.scale)
    torch.cuda.synchronize()
    assert_bits_equal(gather_f32(shards, idx_dev), gout, "1.3B reduced gradients")
    assert not shards[pb.n:].any()
    del pb, args, keep, shards
    _free()


def test_gpt_1p3b_checked_step():
    """The overflow-checked step on the 1.3B list as the benchmark runs it
    (--check-overflow: two passes through the caller's workspace, the range
    far above one resident wave).  A clean step matches the oracle at the
    sampled indices; the next step, with one +inf injected into one rank's
    gradient, raises the flag and leaves every sampled value of master, m, v
    and the replicas as the clean step left it."""
    wl = workloads.gpt_1p3b()
    seed = 4
    pb = Problem(wl, seed)
    rng = np.random.default_rng(seed)
    bad_q, bad_i = int(rng.integers(0, pb.P)), int(rng.integers(0, pb.n))
    idx = sample_indices(pb.n, pb.S, pb.P, seed, extra=[t.offset for t in wl.tensors] + [bad_i],
                         k_random=50_000, around=8)
    idx_dev = torch.from_numpy(idx).to(DEV)
    w, m, v = pb.oracle_state(idx_dev)
    args, keep = zdp.make_step_args(pb.grads, *pb.buffers(), pb.replicas, n=pb.n,
                                    scale=wl.scale, t=1, d_overflow=pb.flag, d_sumsq=pb.sumsq,
                                    check_overflow=True, **HP)
    ws = torch.empty(zdp.zdp_step_workspace_bytes(args), dtype=torch.uint8, device=DEV)
    args.workspace, args.workspace_bytes = ws.data_ptr(), ws.numel()
    rep = None
    for t in (1, 2):
        for q in range(pb.P):
            workloads.fill_grads(pb.grads[q], wl, q, t, seed)
        if t == 2:
            pb.grads[bad_q].view(torch.int16)[bad_i] = 0x7F80  # bf16 +inf
        gs = np.stack([gather_bits(g, idx_dev) for g in pb.grads])
        pb.words.zero_()
        args.t = t
        zdp.zdp_step(args)
        torch.cuda.synchronize()
        # the flag first (on copies: skip=True leaves the state alone), then
        # the step as the flag decides
        _, _, flag = oracle.step_sampled(gs, idx, oracle.BF16, w.copy(), m.copy(), v.copy(),
                                         pb.n, wl.scale, t=t, skip=True, **HP)
        assert flag == (1 if t == 2 else 0)
        assert int(pb.flag.item()) == flag
        _, rep_t, _ = oracle.step_sampled(gs, idx, oracle.BF16, w, m, v, pb.n, wl.scale, t=t,
                                          skip=bool(flag), **HP)
        if not flag:
            rep = rep_t  # a skipped step leaves the replicas as the clean step wrote them
        pb.check(idx, idx_dev, w, m, v, rep, f"1.3B checked t={t}")
    del pb, args, keep, ws
    _free()


def test_gpt_1p3b_unfused_chain():
    """The step's three calls at the 1.3B size, as `bench.py --unfused` runs
    them: reduce-scatter into fp32 shards, AdamW over the whole P*S range,
    all-gather of the new master into the P replicas."""
    wl = workloads.gpt_1p3b()
    seed = 7
    pb = Problem(wl, seed)
    idx = sample_indices(pb.n, pb.S, pb.P, seed, extra=[t.offset for t in wl.tensors],
                         k_random=50_000, around=8)
    idx_dev = torch.from_numpy(idx).to(DEV)
    w, m, v = pb.oracle_state(idx_dev)
    for q in range(pb.P):
        workloads.fill_grads(pb.grads[q], wl, q, 1, seed)
    gs = np.stack([gather_bits(g, idx_dev) for g in pb.grads])
    shards = torch.empty(pb.P * pb.S, dtype=torch.float32, device=DEV)
    zdp.zdp_reduce_scatter(pb.grads, shards, pb.n, pb.P, wl.scale, d_overflow=pb.flag,
                           d_sumsq=pb.sumsq)
    zdp.zdp_adamw_shard(pb.state[0], pb.state[1], pb.state[2], shards, pb.P * pb.S, t=1, **HP)
    zdp.zdp_all_gather(pb.state[0], pb.replicas, pb.n, pb.P)
    torch.cuda.synchronize()
    gout, rep, flag = oracle.step_sampled(gs, idx, oracle.BF16, w, m, v, pb.n, wl.scale, t=1,
                                          **HP)
    assert flag == 0 and int(pb.flag.item()) == 0
    assert_bits_equal(gather_f32(shards, idx_dev), gout, "1.3B unfused reduced gradients")
    pb.check(idx, idx_dev, w, m, v, rep, "1.3B unfused chain")
    del pb, shards
    _free()


def test_gpt_7b_streamed_buckets():
    # fp32 state (79 GB) and 8 replicas (105 GB) resident; each rank's
    # gradients regenerated one 256 MiB bucket at a time by a producer stream
    # into two bucket buffers, while zdp_step (off/len) runs on the previous
    # bucket on a second stream: the ZeRO-2 streamed step, overlapped
    wl = workloads.gpt_7b()
    seed = 4
    pb = Problem(wl, seed, grads=False)
    B = wl.bucket_elems
    idx = sample_indices(pb.n, pb.S, pb.P, seed,
                         extra=list(range(0, pb.n, B)) + [t.offset for t in wl.tensors],
                         k_random=50_000, around=4)
    idx_dev = torch.from_numpy(idx).to(DEV)
    w, m, v = pb.oracle_state(idx_dev)
    ss = streaming.StreamedStep(pb.P, pb.n, B, pb.state[0], pb.state[1], pb.state[2],
                                pb.replicas, scale=wl.scale, d_overflow=pb.flag,
                                d_sumsq=pb.sumsq, **HP)
    prod = SampledProducer(wl, seed, idx, pb.P)
    prod.prepare(ss.bounds)
    prod.step = 0
    ss.run(wl.t0, prod)
    torch.cuda.synchronize()
    gout, rep, flag = oracle.step_sampled(prod.host_values(), idx, oracle.BF16, w, m, v, pb.n,
                                          wl.scale, t=wl.t0, **HP)
    assert flag == 0 and int(pb.flag.item()) == 0
    pb.check(idx, idx_dev, w, m, v, rep, "7B streamed")
    del pb, ss, prod
    _free()


FULL_LIMIT = 1 << 22  # P*n up to which the oracle checks every element


@pytest.mark.parametrize("P", workloads.SWEEP_P)
def test_fp16_sweep_with_overflow_skip(P):
    seed = 5
    for point, n in enumerate(workloads.SWEEP_N):
        wl = workloads.sweep_point(n, P)
        for rep_i, force in ((0, False), (1, True)):
            plan = workloads.injection_plan(seed, 100 * P + point, rep_i, n, P, force=force)
            pb = Problem(wl, seed + point)
            for q in range(P):
                workloads.fill_grads(pb.grads[q], wl, q, rep_i, seed)
            for q, i, bits in plan:
                pb.grads[q].view(torch.int16)[i] = bits - 65536 if bits >= 32768 else bits
            ws = torch.empty(256 + ((n + 8) * 4 + 255) // 256 * 256, dtype=torch.uint8,
                             device=DEV)
            args, keep = zdp.make_step_args(pb.grads, pb.state[0], pb.state[1], pb.state[2],
                                            pb.replicas, n=n, scale=wl.scale, t=wl.t0,
                                            check_overflow=True, d_overflow=pb.flag,
                                            d_sumsq=pb.sumsq, workspace=ws,
                                            workspace_bytes=ws.numel(), **HP)
            if P * n <= FULL_LIMIT:
                idx = np.arange(n, dtype=np.int64)
            else:
                idx = sample_indices(n, pb.S, P, seed + point, extra=[i for _, i, _ in plan],
                                     k_random=20_000, around=8)
            idx_dev = torch.from_numpy(idx).to(DEV)
            w, m, v = pb.oracle_state(idx_dev)
            rep_before = gather_bits(pb.replicas[0], idx_dev)
            gs = np.stack([gather_bits(g, idx_dev) for g in pb.grads])
            zdp.zdp_step(args)
            torch.cuda.synchronize()
            # flag first (sampled: the injected positions are all in the sample)
            _, _, flag = oracle.step_sampled(gs, idx, oracle.FP16, w.copy(), m.copy(), v.copy(),
                                             n, wl.scale, t=wl.t0, skip=True, **HP)
            label = f"P={P} n={n} run={rep_i} injected={len(plan)}"
            assert flag == (1 if plan else 0), label
            assert int(pb.flag.item()) == flag, label
            gout, rep, _ = oracle.step_sampled(gs, idx, oracle.FP16, w, m, v, n, wl.scale,
                                               t=wl.t0, skip=bool(flag), **HP)
            if flag:
                rep = rep_before  # a skipped step leaves the replicas alone
            pb.check(idx, idx_dev, w, m, v, rep, label)
            del pb, args, keep, ws
        _free()
