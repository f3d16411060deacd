"""The step inside a CUDA graph.

A training loop captures its step once and replays it, so every call must be
capturable: the bucketed fused step (its launches carry programmatic stream
serialization), the single-pass checked step (a memset and a cooperative
launch) and the two-pass checked step (a memset and two kernels per bucket).
A replay of the captured call must give the same bits as the same call made
eagerly on the same inputs.
"""

import numpy as np
import pytest
import torch

import oracle
from harness import DeviceStep, assert_bits_equal, random_problem

pytestmark = pytest.mark.gpu


def _eager_and_graph(P, n, gdt, **kw):
    gbits, w, m, v = random_problem(P, n, P + n, gdt)
    rep = np.zeros((P, n), np.uint16)
    dtype = torch.float16 if gdt == oracle.FP16 else torch.bfloat16
    scale = 1.0 / (P * (65536.0 if gdt == oracle.FP16 else 1.0))

    eager = DeviceStep(P, n, dtype)
    eager.load(gbits, w, m, v, rep)
    eager.step(scale, 9, **kw)

    graphed = DeviceStep(P, n, dtype)
    graphed.load(gbits, w, m, v, rep)
    a, keep = graphed.args(scale, 9, **kw)
    from zero_gradient_reduce_gb300 import zdp
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            zdp.zdp_step(a)  # captured, not run
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    # nothing ran during capture
    assert_bits_equal(graphed.state()[0], w, "state before replay")
    g.replay()
    torch.cuda.synchronize()
    return eager, graphed


def _same(a, b, label):
    for x, y, name in zip(a.state(), b.state(), ("master", "m", "v")):
        assert_bits_equal(x, y, f"{label} {name}")
    assert np.array_equal(a.replica_bits(), b.replica_bits()), f"{label} replicas"
    assert int(a.flag.item()) == int(b.flag.item()), f"{label} flag"


@pytest.mark.parametrize("bucket", [0, 100_003])
def test_fused_step_replays_from_a_graph(bucket):
    eager, graphed = _eager_and_graph(8, 1_000_003, oracle.BF16, bucket_elems=bucket)
    _same(eager, graphed, f"fused bucket={bucket}")


@pytest.mark.parametrize("n,bucket", [(200_003, 0), (3_000_001, 700_000)])
def test_checked_step_replays_from_a_graph(n, bucket):
    # n = 200,003 takes the single cooperative launch, 3,000,001 the two passes
    eager, graphed = _eager_and_graph(8, n, oracle.FP16, check_overflow=True,
                                      bucket_elems=bucket)
    _same(eager, graphed, f"checked n={n}")
