"""Checkpoint and resume: a run stopped after k steps and restarted from its
saved state ends bit-identical to a run that never stopped.

The saved state is what the step owns: the fp32 master weight and the two
moments (fp32, or bf16 in the 12-byte variant), plus the step counter t.
Each rank's shard [r*S, min((r+1)*S, n)) is saved on its own.  CS336
Lecture 8 notes ("Parallelism II"), 9.5, describe such checkpoints: each
rank writes only its own share, copied first to host memory and written out
in the background.  Here the copies run on a side stream into pinned host
buffers, ordered after the step by an event.  The restore allocates fresh
device buffers at new addresses.  The replicas are not saved: they are
bf16(master) and zdp_all_gather rebuilds them.
"""

import pytest
import torch

from harness import HP
from zero_gradient_reduce_gb300 import zdp

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")


def _grads(P, n, step, seed):
    g = torch.Generator(device=DEV)
    out = []
    for q in range(P):
        g.manual_seed(seed * 1_000_003 + step * 1009 + q)
        out.append((torch.randn(n, device=DEV, generator=g) * 1e-3).to(torch.bfloat16))
    return out


def _fresh_state(P, n, moments, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    w = torch.randn(n, device=DEV, generator=g) * 0.02
    mdt = torch.float32 if moments == "f32" else torch.bfloat16
    m = torch.zeros(n, dtype=mdt, device=DEV)
    v = torch.zeros(n, dtype=mdt, device=DEV)
    reps = [torch.empty(n, dtype=torch.bfloat16, device=DEV) for _ in range(P)]
    return w, m, v, reps


def _step(P, n, w, m, v, reps, t, moments, seed):
    g = _grads(P, n, t, seed)
    a, keep = zdp.make_step_args(g, w, m, v, reps, n=n, scale=1.0 / P, t=t, moments=moments, **HP)
    zdp.zdp_step(a)


def _save(P, n, w, m, v, t):
    """Per-rank shards of master/m/v copied to pinned host memory on a side stream."""
    S = -(-n // P)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    shards = []
    with torch.cuda.stream(side):
        for r in range(P):
            lo, hi = r * S, min((r + 1) * S, n)
            if lo >= hi:
                shards.append(None)  # a shard that is all padding holds nothing
                continue
            host = [torch.empty(hi - lo, dtype=x.dtype, pin_memory=True) for x in (w, m, v)]
            for h, x in zip(host, (w, m, v)):
                h.copy_(x[lo:hi], non_blocking=True)
            shards.append((lo, hi, host))
    done = torch.cuda.Event()
    done.record(side)
    return {"t": t, "shards": shards, "done": done}


def _restore(P, n, ckpt, moments):
    ckpt["done"].synchronize()
    mdt = torch.float32 if moments == "f32" else torch.bfloat16
    w = torch.full((n,), float("nan"), device=DEV)
    m = torch.full((n,), float("nan"), dtype=mdt, device=DEV)
    v = torch.full((n,), float("nan"), dtype=mdt, device=DEV)
    for entry in ckpt["shards"]:
        if entry is None:
            continue
        lo, hi, host = entry
        for x, h in zip((w, m, v), host):
            x[lo:hi].copy_(h, non_blocking=True)
    reps = [torch.empty(n, dtype=torch.bfloat16, device=DEV) for _ in range(P)]
    zdp.zdp_all_gather(w, reps, n, P)
    return w, m, v, reps, ckpt["t"]


@pytest.mark.parametrize("P,n", [(4, 200_003), (8, 1 << 20), (3, 10)])
@pytest.mark.parametrize("moments", ["f32", "bf16"])
def test_resume_is_bit_identical(P, n, moments):
    k1, k2, seed = 3, 4, 17
    # uninterrupted
    w, m, v, reps = _fresh_state(P, n, moments, seed)
    for t in range(1, k1 + k2 + 1):
        _step(P, n, w, m, v, reps, t, moments, seed)
    torch.cuda.synchronize()
    # interrupted after k1 steps, state saved, device state discarded, restored
    w2, m2, v2, reps2 = _fresh_state(P, n, moments, seed)
    for t in range(1, k1 + 1):
        _step(P, n, w2, m2, v2, reps2, t, moments, seed)
    reps_at_k1 = [r.clone() for r in reps2]
    ckpt = _save(P, n, w2, m2, v2, k1)
    ckpt["done"].synchronize()  # the side-stream copies have read the state
    del w2, m2, v2, reps2
    w3, m3, v3, reps3, t0 = _restore(P, n, ckpt, moments)
    torch.cuda.synchronize()
    for q in range(P):  # the rebuilt replicas are the ones the step wrote
        assert torch.equal(reps3[q].view(torch.int16), reps_at_k1[q].view(torch.int16)), q
    for t in range(t0 + 1, t0 + k2 + 1):
        _step(P, n, w3, m3, v3, reps3, t, moments, seed)
    torch.cuda.synchronize()
    for x, y, name in ((w, w3, "master"), (m, m3, "m"), (v, v3, "v")):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), name
    for q in range(P):
        assert torch.equal(reps[q].view(torch.int16), reps3[q].view(torch.int16)), f"replica {q}"
