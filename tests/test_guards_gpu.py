"""Every call writes its outputs and nothing else.

Each buffer the library sees, input or output, sits inside a larger
allocation filled with a canary byte: 256 guard bytes before it and at
least 256 after.  After each call the test checks three things:
  * every guard byte is intact;
  * the inputs are unchanged;
  * the outputs equal, bit for bit, those of the same call on ordinary
    unguarded tensors.
Output lengths are the documented minimums (master, m, v and the replicas
hold n elements, not P*S), so a write past element n-1 lands in a guard.
Cases cover P in {1, 2, 3, 5, 8, 64}, n from 1 up through several
thousand, pointers shifted by one element (the scalar path), checked and
unchecked steps, the unfused calls, the literal ring, ZeRO++, the quantizer
and the plain copy.
"""

import numpy as np
import pytest
import torch

from harness import HP
from zero_gradient_reduce_gb300 import zdp

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")
G = 256
PAT = 0xA5


class Guarded:
    """`nbytes` bytes at byte offset G + shift of a canary-filled allocation."""

    def __init__(self, nbytes, shift=0):
        self.nbytes, self.off = nbytes, G + shift
        self.buf = torch.full((nbytes + 2 * G + 16,), PAT, dtype=torch.uint8, device=DEV)

    def typed(self, dtype):
        es = torch.empty((), dtype=dtype).element_size()
        assert self.nbytes % es == 0 and self.off % es == 0
        return self.buf[self.off:self.off + self.nbytes].view(dtype)

    def bytes(self):
        return self.buf[self.off:self.off + self.nbytes]

    def guards_intact(self):
        b = self.buf.cpu().numpy()
        return bool((b[:self.off] == PAT).all() and (b[self.off + self.nbytes:] == PAT).all())


def _g(count, dtype, shift_elems=0, fill=None):
    es = torch.empty((), dtype=dtype).element_size()
    gb = Guarded(count * es, shift_elems * es)
    if fill is not None:
        gb.typed(dtype).copy_(fill)
    return gb


def _bf16(rng, count, scale):
    return torch.from_numpy((rng.standard_normal(count) * scale).astype(np.float32)).to(DEV).to(torch.bfloat16)


def _check_all(guarded, inputs_before, what):
    for name, gb in guarded.items():
        assert gb.guards_intact(), f"{what}: guard of {name} overwritten"
    for name, (gb, before) in inputs_before.items():
        assert torch.equal(gb.bytes(), before), f"{what}: input {name} modified"


def _same_bytes(a, b, what):
    assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8)), what


CASES = [(P, n) for P in (1, 2, 3, 5, 8, 64) for n in sorted({1, 7, P + 1, 4097, 20003})]


@pytest.mark.parametrize("P,n", CASES)
@pytest.mark.parametrize("shift,check", [(0, False), (0, True), (1, False)])
def test_step_writes_only_its_outputs(P, n, shift, check):
    rng = np.random.default_rng(P * 100003 + n)
    g_vals = [_bf16(rng, n, 1e-3) for _ in range(P)]
    w0 = torch.from_numpy((rng.standard_normal(n) * 0.02).astype(np.float32)).to(DEV)
    m0 = torch.from_numpy((rng.standard_normal(n) * 1e-4).astype(np.float32)).to(DEV)
    v0 = torch.from_numpy(rng.uniform(0, 1e-6, n).astype(np.float32)).to(DEV)
    # guarded run
    gg = [_g(n, torch.bfloat16, shift, g_vals[q]) for q in range(P)]
    gw, gm, gv = (_g(n, torch.float32, shift, x) for x in (w0, m0, v0))
    gr = [_g(n, torch.bfloat16, shift) for _ in range(P)]
    gflag, gss = Guarded(4), Guarded(8)
    gflag.bytes().zero_()
    gss.bytes().zero_()
    a, keep = zdp.make_step_args([x.typed(torch.bfloat16) for x in gg], gw.typed(torch.float32),
                                 gm.typed(torch.float32), gv.typed(torch.float32),
                                 [x.typed(torch.bfloat16) for x in gr], n=n, scale=1.0 / P, t=3,
                                 check_overflow=check, d_overflow=gflag.typed(torch.int32),
                                 d_sumsq=gss.typed(torch.float64), **HP)
    guarded = {f"grads[{q}]": x for q, x in enumerate(gg)}
    guarded.update({"master": gw, "m": gm, "v": gv, "flag": gflag, "sumsq": gss})
    guarded.update({f"replicas[{q}]": x for q, x in enumerate(gr)})
    if check:
        gws = Guarded(zdp.zdp_step_workspace_bytes(a))
        a.workspace, a.workspace_bytes = gws.bytes().data_ptr(), gws.nbytes
        guarded["workspace"] = gws
    inputs = {f"grads[{q}]": (x, x.bytes().clone()) for q, x in enumerate(gg)}
    zdp.zdp_step(a)
    torch.cuda.synchronize()
    _check_all(guarded, inputs, f"step P={P} n={n} shift={shift} check={check}")
    # the same call on ordinary tensors
    rw, rm, rv = w0.clone(), m0.clone(), v0.clone()
    rr = [torch.zeros(n, dtype=torch.bfloat16, device=DEV) for _ in range(P)]
    words = torch.zeros(16, dtype=torch.uint8, device=DEV)
    rg = [x.clone() for x in g_vals]  # held: the call only records their addresses
    ra, rkeep = zdp.make_step_args(rg, rw, rm, rv, rr, n=n,
                                   scale=1.0 / P, t=3, check_overflow=check,
                                   d_overflow=words[0:4].view(torch.int32),
                                   d_sumsq=words[8:16].view(torch.float64), **HP)
    ws = None
    if check:
        ws = torch.empty(zdp.zdp_step_workspace_bytes(ra), dtype=torch.uint8, device=DEV)
        ra.workspace, ra.workspace_bytes = ws.data_ptr(), ws.numel()
    zdp.zdp_step(ra)
    torch.cuda.synchronize()
    label = f"P={P} n={n} shift={shift} check={check}"
    _same_bytes(gw.typed(torch.float32), rw, label + " master")
    _same_bytes(gm.typed(torch.float32), rm, label + " m")
    _same_bytes(gv.typed(torch.float32), rv, label + " v")
    for q in range(P):
        _same_bytes(gr[q].typed(torch.bfloat16), rr[q], label + f" replica {q}")
    _same_bytes(gflag.bytes(), words[0:4], label + " flag")
    # the sum of squares adds in a different order on different launch shapes
    got = float(gss.typed(torch.float64).item())
    want = float(words[8:16].view(torch.float64).item())
    assert abs(got - want) <= 1e-12 * abs(want), (label, got, want)


@pytest.mark.parametrize("P,n", [(1, 1), (3, 7), (5, 4097), (8, 20003), (64, 20003)])
@pytest.mark.parametrize("shift", [0, 1])
def test_unfused_calls_write_only_their_outputs(P, n, shift):
    rng = np.random.default_rng(n + P)
    S = -(-n // P)
    g_vals = [_bf16(rng, n, 1e-3) for _ in range(P)]
    gg = [_g(n, torch.bfloat16, shift, g_vals[q]) for q in range(P)]
    gsh = _g(P * S, torch.float32, shift)
    gflag = Guarded(4)
    gflag.bytes().zero_()
    inputs = {f"grads[{q}]": (x, x.bytes().clone()) for q, x in enumerate(gg)}
    zdp.zdp_reduce_scatter([x.typed(torch.bfloat16) for x in gg], gsh.typed(torch.float32), n, P,
                           1.0 / P, d_overflow=gflag.typed(torch.int32))
    torch.cuda.synchronize()
    guarded = {"shards": gsh, "flag": gflag, **{f"grads[{q}]": x for q, x in enumerate(gg)}}
    _check_all(guarded, inputs, f"reduce_scatter P={P} n={n}")
    ref = torch.empty(P * S, dtype=torch.float32, device=DEV)
    rg = [x.clone() for x in g_vals]
    zdp.zdp_reduce_scatter(rg, ref, n, P, 1.0 / P)
    torch.cuda.synchronize()
    _same_bytes(gsh.typed(torch.float32), ref, "shards")

    # AdamW on the whole padded range of shards, in place on guarded state
    w0 = torch.from_numpy((rng.standard_normal(P * S) * 0.02).astype(np.float32)).to(DEV)
    gw = _g(P * S, torch.float32, shift, w0)
    gm = _g(P * S, torch.float32, shift, torch.zeros(P * S, device=DEV))
    gv = _g(P * S, torch.float32, shift, torch.zeros(P * S, device=DEV))
    shards_before = gsh.bytes().clone()
    zdp.zdp_adamw_shard(gw.typed(torch.float32), gm.typed(torch.float32), gv.typed(torch.float32),
                        gsh.typed(torch.float32), P * S, t=1, **HP)
    torch.cuda.synchronize()
    _check_all({"master": gw, "m": gm, "v": gv, "shards": gsh},
               {"shards": (gsh, shards_before)}, f"adamw_shard P={P} n={n}")
    rw, rm, rv = w0.clone(), torch.zeros_like(w0), torch.zeros_like(w0)
    zdp.zdp_adamw_shard(rw, rm, rv, ref, P * S, t=1, **HP)
    torch.cuda.synchronize()
    _same_bytes(gw.typed(torch.float32), rw, "adamw master")
    _same_bytes(gm.typed(torch.float32), rm, "adamw m")

    # all-gather of the first n master values into guarded replicas
    gr = [_g(n, torch.bfloat16, shift) for _ in range(P)]
    master_before = gw.bytes().clone()
    zdp.zdp_all_gather(gw.typed(torch.float32), [x.typed(torch.bfloat16) for x in gr], n, P)
    torch.cuda.synchronize()
    _check_all({"master": gw, **{f"replicas[{q}]": x for q, x in enumerate(gr)}},
               {"master": (gw, master_before)}, f"all_gather P={P} n={n}")
    want = rw[:n].to(torch.bfloat16)
    for q in range(P):
        _same_bytes(gr[q].typed(torch.bfloat16), want, f"replica {q}")


@pytest.mark.parametrize("P,n", [(2, 7), (3, 4097), (8, 20003)])
def test_ring_step_writes_only_its_outputs(P, n):
    rng = np.random.default_rng(7 * n + P)
    g_vals = [_bf16(rng, n, 1e-3) for _ in range(P)]
    w0 = torch.from_numpy((rng.standard_normal(n) * 0.02).astype(np.float32)).to(DEV)
    gg = [_g(n, torch.bfloat16, 0, g_vals[q]) for q in range(P)]
    gw = _g(n, torch.float32, 0, w0)
    gm = _g(n, torch.float32, 0, torch.zeros(n, device=DEV))
    gv = _g(n, torch.float32, 0, torch.zeros(n, device=DEV))
    gr = [_g(n, torch.bfloat16) for _ in range(P)]
    a, keep = zdp.make_step_args([x.typed(torch.bfloat16) for x in gg], gw.typed(torch.float32),
                                 gm.typed(torch.float32), gv.typed(torch.float32),
                                 [x.typed(torch.bfloat16) for x in gr], n=n, scale=1.0 / P, t=1,
                                 **HP)
    gws = Guarded(zdp.zdp_step_ring_workspace_bytes(a))
    a.workspace, a.workspace_bytes = gws.bytes().data_ptr(), gws.nbytes
    inputs = {f"grads[{q}]": (x, x.bytes().clone()) for q, x in enumerate(gg)}
    zdp.zdp_step_ring(a)
    torch.cuda.synchronize()
    guarded = {"master": gw, "m": gm, "v": gv, "workspace": gws}
    guarded.update({f"replicas[{q}]": x for q, x in enumerate(gr)})
    _check_all(guarded, inputs, f"ring P={P} n={n}")
    rw, rm, rv = w0.clone(), torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
    rr = [torch.zeros(n, dtype=torch.bfloat16, device=DEV) for _ in range(P)]
    rg = [x.clone() for x in g_vals]
    ra, rkeep = zdp.make_step_args(rg, rw, rm, rv, rr, n=n, scale=1.0 / P, t=1, **HP)
    zdp.zdp_step(ra)  # the ring gives the fused step's bits
    torch.cuda.synchronize()
    _same_bytes(gw.typed(torch.float32), rw, "ring master")
    for q in range(P):
        _same_bytes(gr[q].typed(torch.bfloat16), rr[q], f"ring replica {q}")


@pytest.mark.parametrize("P,n", [(1, 1), (3, 255), (8, 256 * 9 + 17), (16, 20003)])
def test_zpp_and_quantizer_write_only_their_outputs(P, n):
    rng = np.random.default_rng(11 * n + P)
    nb = -(-n // 256)
    x = torch.from_numpy((rng.standard_normal(n) * 1e-3).astype(np.float32)).to(DEV)
    gx = _g(n, torch.float32, 0, x)
    gq, gs = _g(n, torch.int8), _g(nb, torch.float32)
    x_before = gx.bytes().clone()
    zdp.zdp_quantize_blocks(gx.typed(torch.float32), zdp.ZDP_F32, n, gq.typed(torch.int8),
                            gs.typed(torch.float32))
    torch.cuda.synchronize()
    _check_all({"x": gx, "q": gq, "scales": gs}, {"x": (gx, x_before)}, f"quantize n={n}")
    gout = _g(n, torch.bfloat16)
    q_before, s_before = gq.bytes().clone(), gs.bytes().clone()
    zdp.zdp_dequantize_blocks(gq.typed(torch.int8), gs.typed(torch.float32), n,
                              gout.typed(torch.bfloat16))
    torch.cuda.synchronize()
    _check_all({"q": gq, "scales": gs, "out": gout},
               {"q": (gq, q_before), "scales": (gs, s_before)}, f"dequantize n={n}")

    codes = [torch.from_numpy(rng.integers(-127, 128, n).astype(np.int8)).to(DEV) for _ in range(P)]
    scales = [torch.from_numpy(rng.uniform(1e-6, 1e-5, nb).astype(np.float32)).to(DEV)
              for _ in range(P)]
    g_q = [_g(n, torch.int8, 0, codes[q]) for q in range(P)]
    g_s = [_g(nb, torch.float32, 0, scales[q]) for q in range(P)]
    w0 = torch.from_numpy((rng.standard_normal(n) * 0.02).astype(np.float32)).to(DEV)
    gw = _g(n, torch.float32, 0, w0)
    gm = _g(n, torch.float32, 0, torch.zeros(n, device=DEV))
    gv = _g(n, torch.float32, 0, torch.zeros(n, device=DEV))
    grq = [_g(n, torch.int8) for _ in range(P)]
    grs = [_g(nb, torch.float32) for _ in range(P)]
    a, keep = zdp.make_zpp_args([t.typed(torch.int8) for t in g_q],
                                [t.typed(torch.float32) for t in g_s], gw.typed(torch.float32),
                                gm.typed(torch.float32), gv.typed(torch.float32),
                                [t.typed(torch.int8) for t in grq],
                                [t.typed(torch.float32) for t in grs], n=n, scale=1.0 / P, t=1,
                                **HP)
    inputs = {f"codes[{q}]": (t, t.bytes().clone()) for q, t in enumerate(g_q)}
    inputs.update({f"grad_scales[{q}]": (t, t.bytes().clone()) for q, t in enumerate(g_s)})
    zdp.zdp_step_zpp(a)
    torch.cuda.synchronize()
    guarded = {"master": gw, "m": gm, "v": gv}
    guarded.update({f"rq[{q}]": t for q, t in enumerate(grq)})
    guarded.update({f"rs[{q}]": t for q, t in enumerate(grs)})
    _check_all(guarded, inputs, f"zpp P={P} n={n}")
    rw, rm, rv = w0.clone(), torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
    rrq = [torch.zeros(n, dtype=torch.int8, device=DEV) for _ in range(P)]
    rrs = [torch.zeros(nb, dtype=torch.float32, device=DEV) for _ in range(P)]
    rc, rsc = [c.clone() for c in codes], [x.clone() for x in scales]
    ra, rkeep = zdp.make_zpp_args(rc, rsc, rw, rm, rv, rrq, rrs, n=n, scale=1.0 / P, t=1, **HP)
    zdp.zdp_step_zpp(ra)
    torch.cuda.synchronize()
    _same_bytes(gw.typed(torch.float32), rw, "zpp master")
    for q in range(P):
        _same_bytes(grq[q].typed(torch.int8), rrq[q], f"zpp replica {q}")
        _same_bytes(grs[q].typed(torch.float32), rrs[q], f"zpp replica scales {q}")


@pytest.mark.parametrize("nbytes", [16, 4096 + 16, (1 << 24) + 48, 3 * (1 << 26)])
def test_copy_is_exact_and_stays_in_bounds(nbytes):
    src = Guarded(nbytes)
    src.bytes().copy_(torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=DEV))
    dst = Guarded(nbytes)
    before = src.bytes().clone()
    zdp.zdp_copy(dst.bytes(), src.bytes(), nbytes)
    torch.cuda.synchronize()
    _check_all({"dst": dst, "src": src}, {"src": (src, before)}, f"copy {nbytes}")
    assert torch.equal(dst.bytes(), before)
