"""zdp_step with its gradients in pinned host memory, as the benchmark's
end-to-end leg calls it: the kernel reads the P gradient buffers straight
over the host link (GB300 maps pinned host memory into the GPU's address
space), with no staging copy.  The result must equal the same step on
device copies of the gradients bit for bit, and the oracle at sampled
indices."""

import gc

import numpy as np
import pytest
import torch

import oracle
from harness import HP, assert_bf16_close, assert_bits_equal, assert_state_close, bits_of
from zero_gradient_reduce_gb300 import workloads, zdp

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")


def _run(grads, wl, seed, moments):
    P, n = wl.P, wl.n
    S = -(-n // P)
    st = torch.empty(3, P * S, dtype=torch.float32, device=DEV)
    workloads.fill_state(st[0], st[1], st[2], wl, seed)
    w, m, v = st[0], st[1], st[2]
    if moments == "bf16":
        m, v = m.to(torch.bfloat16), v.to(torch.bfloat16)
    reps = [torch.zeros(n, dtype=torch.bfloat16, device=DEV) for _ in range(P)]
    words = torch.zeros(16, dtype=torch.uint8, device=DEV)
    a, keep = zdp.make_step_args(grads, w, m, v, reps, n=n, scale=wl.scale, t=3,
                                 d_overflow=words[0:4].view(torch.int32),
                                 d_sumsq=words[8:16].view(torch.float64), moments=moments, **HP)
    zdp.zdp_step(a)
    torch.cuda.synchronize()
    del a, keep
    return w, m, v, reps, words


@pytest.mark.parametrize("moments", ["f32", "bf16"])
def test_step_on_pinned_host_gradients(moments):
    wl = workloads.gpt2_small()
    P, n, seed = wl.P, wl.n, 6
    S = -(-n // P)
    dev_grads = [workloads.fill_grads(torch.empty(n, dtype=torch.bfloat16, device=DEV), wl, q, 1,
                                      seed) for q in range(P)]
    host_grads = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(P)]
    for q in range(P):
        host_grads[q].copy_(dev_grads[q])
    torch.cuda.synchronize()

    # the oracle's inputs at sampled indices, before either step
    rng = np.random.default_rng(seed)
    pts = {0, n - 1} | {r * S + d for r in range(1, P) for d in range(-8, 8)}
    pts |= set(rng.integers(0, n, 20_000).tolist())
    idx = np.array(sorted(i for i in pts if 0 <= i < n), np.int64)
    idx_dev = torch.from_numpy(idx).to(DEV)
    st0 = torch.empty(3, P * S, dtype=torch.float32, device=DEV)
    workloads.fill_state(st0[0], st0[1], st0[2], wl, seed)
    ow = st0[0].index_select(0, idx_dev).cpu().numpy().copy()
    if moments == "f32":
        om = st0[1].index_select(0, idx_dev).cpu().numpy().copy()
        ov = st0[2].index_select(0, idx_dev).cpu().numpy().copy()
    else:
        om = bits_of(st0[1].index_select(0, idx_dev).to(torch.bfloat16)).copy()
        ov = bits_of(st0[2].index_select(0, idx_dev).to(torch.bfloat16)).copy()
    del st0
    gs = np.stack([bits_of(g.index_select(0, idx_dev)) for g in dev_grads])

    hw, hm, hv, hreps, hwords = _run(host_grads, wl, seed, moments)
    dw, dm, dv, dreps, dwords = _run(dev_grads, wl, seed, moments)

    # host-read step == device-read step, every element
    for name, a, b in (("master", hw, dw), ("m", hm, dm), ("v", hv, dv)):
        ai = a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16)
        bi = b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16)
        assert int((ai != bi).sum().item()) == 0, f"{moments}: {name} differs"
    for q in range(P):
        assert torch.equal(hreps[q].view(torch.int16), dreps[q].view(torch.int16)), f"replica {q}"
    assert int(hwords[0:4].view(torch.int32).item()) == 0
    assert int(dwords[0:4].view(torch.int32).item()) == 0
    hs, ds = float(hwords[8:16].view(torch.float64).item()), float(dwords[8:16].view(torch.float64).item())
    assert abs(hs - ds) <= 1e-12 * ds

    # and the oracle, at the sampled indices
    gout, rep, flag = oracle.step_sampled(gs, idx, oracle.BF16, ow, om, ov, n, wl.scale, t=3,
                                          moments=moments, **HP)
    assert flag == 0
    label = f"host gradients, {moments} moments"
    assert_state_close(hw.index_select(0, idx_dev).cpu().numpy(), ow, label + " master")
    if moments == "f32":
        assert_state_close(hm.index_select(0, idx_dev).cpu().numpy(), om, label + " m")
        assert_state_close(hv.index_select(0, idx_dev).cpu().numpy(), ov, label + " v")
    else:
        assert_bits_equal(bits_of(hm.index_select(0, idx_dev)), om, label + " m")
        assert_bits_equal(bits_of(hv.index_select(0, idx_dev)), ov, label + " v")
    for q in (0, P - 1):
        assert_bf16_close(bits_of(hreps[q].index_select(0, idx_dev)), rep, f"{label} replica {q}")
    del host_grads, dev_grads
    gc.collect()
    torch.cuda.empty_cache()
