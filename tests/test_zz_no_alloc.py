"""zdp_step_noalloc: the overflow-checked step for callers that cannot allocate.

Some callers cannot call cudaMalloc: a plug-in running inside a framework
whose caching allocator owns the device memory, or a step loop that must not
allocate because cudaMalloc/cudaFree synchronise the device.  For them the
library keeps the checked step's scratch, in either of its forms, in its own
static device array (ZDP_NOALLOC_MAX_LEN elements), so the caller passes only
inputs and outputs.

These tests call it through the C ABI and compare it with zdp_step run with a
caller workspace: identical results on consecutive calls (the shared scratch
keeps the previous call's contents, and a raised flag from one call must not
leak into the next), and a clear error for ranges beyond the limit.  This file
is named to be collected last.
"""

import numpy as np
import pytest

from zero_gradient_reduce_gb300 import zdp

FAKE = 1 << 40  # never dereferenced: the size check rejects the call first


def test_rejects_ranges_beyond_the_static_scratch():
    grads = [FAKE + q * (1 << 30) for q in range(2)]
    reps = [FAKE + (8 + q) * (1 << 30) for q in range(2)]
    n = zdp.ZDP_NOALLOC_MAX_LEN + 1
    a, keep = zdp.make_step_args(grads, FAKE + (16 << 30), FAKE + (20 << 30), FAKE + (24 << 30),
                                 reps, n=n, scale=0.5, t=1, lr=1e-3, b1=0.9, b2=0.95, eps=1e-8,
                                 wd=0.0)
    with pytest.raises(zdp.ZdpError) as e:
        zdp.zdp_step_noalloc(a, stream=0)
    assert e.value.status == zdp.ZDP_ERR_INVALID
    assert "ZDP_NOALLOC_MAX_LEN" in str(e.value)


def _pair(P, n, seed):
    import torch
    from harness import DeviceStep, random_problem

    import oracle

    gbits, w, m, v = random_problem(P, n, seed, oracle.FP16)
    a = DeviceStep(P, n, torch.float16)
    b = DeviceStep(P, n, torch.float16)
    for d in (a, b):
        d.load(gbits, w, m, v, np.full((P, n), 0x3F80, np.uint16))
    return a, b


def _new_grads(devs, P, n, seed, inject=None):
    import torch
    from harness import tensor_from_bits

    rng = np.random.default_rng(seed)
    g = (rng.standard_normal((P, n)) * 1e-3 * 65536.0).astype(np.float16).view(np.uint16)
    if inject is not None:
        q, i = inject
        g[q, i] = 0x7C00  # +inf
    for d in devs:
        for q in range(P):
            d.grads[q].copy_(tensor_from_bits(g[q], torch.float16, "cpu"))


def _same(a, b, label):
    from harness import assert_bf16_close, assert_state_close

    for x, y, name in zip(a.state(), b.state(), ("master", "m", "v")):
        assert_state_close(x, y, f"{label} {name}")
    assert_bf16_close(a.replica_bits(), b.replica_bits(), f"{label} replicas")
    assert int(a.flag.item()) == int(b.flag.item()), f"{label} flag"
    assert float(a.sumsq.item()) == pytest.approx(float(b.sumsq.item()), rel=1e-9, abs=0.0)


def _run(d, noalloc, t, off=0, length=None, bucket=0):
    import torch

    d.flag.zero_()
    d.sumsq.zero_()
    scale = 1.0 / (d.P * 65536.0)
    if noalloc:
        args, keep = d.args(scale, t, off=off, length=length, bucket_elems=bucket)
        zdp.zdp_step_noalloc(args)
    else:
        args, keep = d.args(scale, t, off=off, length=length, bucket_elems=bucket,
                            check_overflow=True)
        zdp.zdp_step(args)
    torch.cuda.synchronize()


@pytest.mark.gpu
def test_matches_the_workspace_step_on_consecutive_calls():
    P, n = 8, 3_000_017
    ref, new = _pair(P, n, seed=21)
    # call 1: an infinity in rank 3's gradient -> both skip the update
    _new_grads((ref, new), P, n, seed=22, inject=(3, 1_234_567))
    _run(ref, False, 1)
    _run(new, True, 1)
    assert int(new.flag.item()) == 1
    _same(ref, new, "call 1")
    # call 2: clean gradients -> both update; a stale flag in the shared
    # scratch would make the no-allocation call skip here
    _new_grads((ref, new), P, n, seed=23)
    _run(ref, False, 1)
    _run(new, True, 1)
    assert int(new.flag.item()) == 0
    _same(ref, new, "call 2")
    # call 3: a ragged sub-range walked in buckets
    _new_grads((ref, new), P, n, seed=24)
    _run(ref, False, 2, off=1_000_003, length=1_500_001, bucket=300_007)
    _run(new, True, 2, off=1_000_003, length=1_500_001, bucket=300_007)
    _same(ref, new, "call 3")


@pytest.mark.gpu
def test_largest_accepted_range():
    P, n = 2, zdp.ZDP_NOALLOC_MAX_LEN
    ref, new = _pair(P, n, seed=31)
    for t in (1, 2):
        _new_grads((ref, new), P, n, seed=32 + t)
        _run(ref, False, t)
        _run(new, True, t)
        _same(ref, new, f"max range, call {t}")


@pytest.mark.gpu
@pytest.mark.parametrize("coop", ["1", "0"])
def test_small_aligned_range_in_both_forms(coop, monkeypatch):
    # About 100K elements with 16-byte aligned buffers fit one resident wave,
    # so zdp_step picks the single cooperative launch, which keeps its flag and
    # barrier counter in the first bytes of the static scratch; ZDP_COOP=0
    # forces the two passes instead.  Two calls in a row: an infinity (the
    # update is skipped), then clean gradients (a flag or counter left in the
    # scratch by the first call would spoil the second).
    monkeypatch.setenv("ZDP_COOP", coop)
    P, n = 4, 100_000
    ref, new = _pair(P, n, seed=41)
    _new_grads((ref, new), P, n, seed=42, inject=(1, 54_321))
    _run(ref, False, 1)
    _run(new, True, 1)
    assert int(new.flag.item()) == 1
    _same(ref, new, f"coop={coop} call 1")
    _new_grads((ref, new), P, n, seed=43)
    _run(ref, False, 1)
    _run(new, True, 1)
    assert int(new.flag.item()) == 0
    _same(ref, new, f"coop={coop} call 2")
