"""ZeRO-2 streaming (CS336 Lecture 7 notes, 8.2 items 1-4: each bucket's
gradients are reduce-scattered as soon as the backward pass produces them,
then freed, and every rank updates the shard it owns; 6.4: buckets overlapped
with the backward pass).  A producer stream writes each bucket's P gradient
slices into one of two bucket buffers while zdp_step runs on the previous
bucket on a second stream (zero_gradient_reduce_gb300.streaming).

Checked two ways: against the oracle at sampled global indices (every bucket,
shard and tensor boundary with neighbours, and random elements) over
consecutive steps of the GPT-2-small-shaped model, and against one
whole-model zdp_step call, bit for bit, on flat models with ragged buckets.
Ownership is global, so no interleaving of the two streams may change a bit.
"""

import numpy as np
import pytest
import torch

import oracle
from harness import HP, SampledProducer, assert_bits_equal, bits_of
from test_parity_full_gpu import Problem, _free, sample_indices
from zero_gradient_reduce_gb300 import streaming, workloads, zdp

pytestmark = pytest.mark.gpu


def test_gpt2_small_streamed_on_two_streams_matches_the_oracle():
    wl = workloads.gpt2_small()
    seed = 6
    pb = Problem(wl, seed, grads=False)
    B = wl.bucket_elems
    idx = sample_indices(pb.n, pb.S, pb.P, seed,
                         extra=list(range(0, pb.n, B)) + [t.offset for t in wl.tensors],
                         k_random=30_000, around=8)
    idx_dev = torch.from_numpy(idx).to("cuda")
    w, m, v = pb.oracle_state(idx_dev)
    ss = streaming.StreamedStep(pb.P, pb.n, B, pb.state[0], pb.state[1], pb.state[2],
                                pb.replicas, scale=wl.scale, d_overflow=pb.flag,
                                d_sumsq=pb.sumsq, **HP)
    assert len(ss.bounds) > 2
    # the bucket-wise generator the overlap benchmark uses as its producer
    prod = SampledProducer(wl, seed, idx, pb.P, fill=workloads.fill_bucket_grads)
    prod.prepare(ss.bounds)
    for t in (1, 2, 3):
        prod.step = t
        pb.words.zero_()
        ss.run(t, prod)
        torch.cuda.synchronize()
        gout, rep, flag = oracle.step_sampled(prod.host_values(), idx, oracle.BF16, w, m, v,
                                              pb.n, wl.scale, t=t, **HP)
        assert flag == 0 and int(pb.flag.item()) == 0
        pb.check(idx, idx_dev, w, m, v, rep, f"gpt2 two streams t={t}")
    del pb, ss, prod
    _free()


@pytest.mark.parametrize("P,n,bucket,nbuf", [(8, 50_000_017, 4_000_037, 2),
                                             (4, 9_999_991, 1_000_003, 2),
                                             (3, 3_000_001, 999_999, 3)])
def test_streamed_buckets_on_two_streams_equal_one_call(P, n, bucket, nbuf):
    wl = workloads.Workload(f"flat_{n}_p{P}", P=P, n=n, tensors=workloads._flat(n), t0=3)
    seed = 11
    S = -(-n // P)

    def state():
        st = [torch.empty(P * S, dtype=torch.float32, device="cuda") for _ in range(3)]
        workloads.fill_state(st[0], st[1], st[2], wl, seed)
        reps = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
        return st, reps, torch.zeros(16, dtype=torch.uint8, device="cuda")

    # reference: every rank's whole gradient resident, one call
    grads = [workloads.fill_grads(torch.empty(n, dtype=torch.bfloat16, device="cuda"), wl, q,
                                  0, seed) for q in range(P)]
    st_ref, reps_ref, words_ref = state()
    a, keep = zdp.make_step_args(grads, st_ref[0], st_ref[1], st_ref[2], reps_ref, n=n,
                                 scale=wl.scale, t=wl.t0,
                                 d_overflow=words_ref[0:4].view(torch.int32),
                                 d_sumsq=words_ref[8:16].view(torch.float64), **HP)
    zdp.zdp_step(a)
    torch.cuda.synchronize()

    # streamed: the producer copies each bucket's slice of the resident gradients
    st, reps, words = state()
    ss = streaming.StreamedStep(P, n, bucket, st[0], st[1], st[2], reps, scale=wl.scale,
                                d_overflow=words[0:4].view(torch.int32),
                                d_sumsq=words[8:16].view(torch.float64), buffers=nbuf, **HP)

    def produce(views, lo, hi):
        for q in range(P):
            views[q].copy_(grads[q][lo:hi])

    ss.run(wl.t0, produce)
    torch.cuda.synchronize()
    assert len(ss.bounds) > nbuf
    for x, y, name in zip(st, st_ref, ("master", "m", "v")):
        assert_bits_equal(x[:n].cpu().numpy(), y[:n].cpu().numpy(), f"streamed {name}")
    for q in range(P):
        assert np.array_equal(bits_of(reps[q]), bits_of(reps_ref[q])), f"replica {q}"
    assert int(words[0:4].view(torch.int32).item()) == int(words_ref[0:4].view(torch.int32).item())
    s_ref = float(words_ref[8:16].view(torch.float64).item())
    assert abs(float(words[8:16].view(torch.float64).item()) - s_ref) <= 1e-9 * s_ref


def test_streamed_fp16_gradients_and_bf16_moments_equal_one_call():
    # the driver's other storage types: fp16 gradients (loss-scaled) and the
    # 12-byte state (bf16 m and v), three bucket buffers
    P, n, bucket = 4, 5_000_011, 700_001
    wl = workloads.Workload(f"flat_{n}_p{P}_fp16", P=P, n=n, tensors=workloads._flat(n),
                            grad_dtype="fp16", fp16_loss_scale=2.0 ** 16, t0=5)
    seed = 13
    S = -(-n // P)
    grads = [workloads.fill_grads(torch.empty(n, dtype=torch.float16, device="cuda"), wl, q,
                                  0, seed) for q in range(P)]

    def state():
        st = torch.empty(3, P * S, dtype=torch.float32, device="cuda")
        workloads.fill_state(st[0], st[1], st[2], wl, seed)
        mv = st[1:].to(torch.bfloat16)
        reps = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
        return st[0].clone(), mv[0], mv[1], reps, torch.zeros(16, dtype=torch.uint8, device="cuda")

    w0, m0, v0, r0, k0 = state()
    a, keep = zdp.make_step_args(grads, w0, m0, v0, r0, n=n, scale=wl.scale, t=wl.t0,
                                 d_overflow=k0[0:4].view(torch.int32), moments="bf16", **HP)
    zdp.zdp_step(a)
    w1, m1, v1, r1, k1 = state()
    ss = streaming.StreamedStep(P, n, bucket, w1, m1, v1, r1, scale=wl.scale,
                                grad_dtype=torch.float16, moments="bf16",
                                d_overflow=k1[0:4].view(torch.int32), buffers=3, **HP)

    def produce(views, lo, hi):
        for q in range(P):
            views[q].copy_(grads[q][lo:hi])

    ss.run(wl.t0, produce)
    torch.cuda.synchronize()
    assert_bits_equal(w1[:n].cpu().numpy(), w0[:n].cpu().numpy(), "streamed master")
    assert np.array_equal(bits_of(m1[:n]), bits_of(m0[:n])) and np.array_equal(bits_of(v1[:n]), bits_of(v0[:n]))
    for q in range(P):
        assert np.array_equal(bits_of(r1[q]), bits_of(r0[q])), f"replica {q}"
    assert int(k1[0:4].view(torch.int32).item()) == int(k0[0:4].view(torch.int32).item()) == 0
