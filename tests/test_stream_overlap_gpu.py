"""ZeRO-2-style streaming (CS336 Lecture 7 notes, 8.2: gradients reduced bucket by
bucket as the backward pass produces them, and freed): a producer stream writes
each bucket's P gradient slices into one of two bucket buffers while zdp_step
runs on the previous bucket on a second stream.  Events order the two streams
(ready: producer -> step; done: step -> producer before the buffer is reused).
Ownership is global, so the streamed step must equal one whole-model call bit
for bit, whatever the interleaving."""

import numpy as np
import pytest
import torch

from harness import HP, assert_bits_equal, bits_of
from zero_gradient_reduce_gb300 import workloads, zdp

pytestmark = pytest.mark.gpu


def _state(wl, seed):
    P, n = wl.P, wl.n
    S = -(-n // P)
    st = [torch.empty(P * S, dtype=torch.float32, device="cuda") for _ in range(3)]
    workloads.fill_state(st[0], st[1], st[2], wl, seed)
    reps = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    words = torch.zeros(16, dtype=torch.uint8, device="cuda")
    return st, reps, words


@pytest.mark.parametrize("P,n,bucket", [(8, 50_000_017, 4_000_037), (4, 9_999_991, 1_000_003)])
def test_streamed_buckets_on_two_streams_equal_one_call(P, n, bucket):
    wl = workloads.Workload(f"flat_{n}_p{P}", P=P, n=n, tensors=workloads._flat(n), t0=3)
    seed = 11
    # reference: every rank's whole gradient resident, one call
    grads = [workloads.fill_grads(torch.empty(n, dtype=torch.bfloat16, device="cuda"), wl, q,
                                  0, seed) for q in range(P)]
    st_ref, reps_ref, words_ref = _state(wl, seed)
    a, keep = zdp.make_step_args(grads, st_ref[0], st_ref[1], st_ref[2], reps_ref, n=n,
                                 scale=wl.scale, t=wl.t0, d_overflow=words_ref[0:4].view(torch.int32),
                                 **HP)
    zdp.zdp_step(a)
    torch.cuda.synchronize()

    # streamed: two bucket buffers, producer and step on separate streams
    st, reps, words = _state(wl, seed)
    bufs = [[torch.empty(bucket, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
            for _ in range(2)]
    producer, stepper = torch.cuda.Stream(), torch.cuda.Stream()
    bounds = [(lo, min(n, lo + bucket)) for lo in range(0, n, bucket)]
    ready = [torch.cuda.Event() for _ in bounds]
    done = [torch.cuda.Event() for _ in bounds]
    keep_all = []
    for b, (lo, hi) in enumerate(bounds):
        buf = bufs[b % 2]
        with torch.cuda.stream(producer):
            if b >= 2:
                producer.wait_event(done[b - 2])  # the step on this buffer has finished
            for q in range(P):  # the gradient's slice [lo, hi), as the full tensor holds it
                buf[q][:hi - lo].copy_(grads[q][lo:hi])
            ready[b].record(producer)
        stepper.wait_event(ready[b])
        sa, sk = zdp.make_step_args([x[:hi - lo] for x in buf], st[0], st[1], st[2], reps, n=n,
                                    scale=wl.scale, t=wl.t0, off=lo, length=hi - lo,
                                    d_overflow=words[0:4].view(torch.int32), **HP)
        keep_all.append((sa, sk))
        zdp.zdp_step(sa, stepper)
        done[b].record(stepper)
    torch.cuda.synchronize()
    assert len(bounds) > 2
    for x, y, name in zip(st, st_ref, ("master", "m", "v")):
        assert_bits_equal(x[:n].cpu().numpy(), y[:n].cpu().numpy(), f"streamed {name}")
    for q in range(P):
        assert np.array_equal(bits_of(reps[q]), bits_of(reps_ref[q])), f"replica {q}"
    assert int(words[0:4].view(torch.int32).item()) == int(words_ref[0:4].view(torch.int32).item())
