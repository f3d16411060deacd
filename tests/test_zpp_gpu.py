"""ZeRO++ on the GPU against the oracle (Fudan MLSys ch. 9, 9.4.3): block int8
quantization and dequantization, and the step with quantized gradients in and
quantized replicas out, element by element, including ragged ends, shard
boundaries inside blocks, sub-ranges, bf16 moments and the 1.3B model."""

import numpy as np
import pytest
import torch

import oracle
from harness import HP, assert_bits_equal, assert_state_close, bits_of
from zero_gradient_reduce_gb300 import workloads, zdp

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")


def _i8(t):
    return t.cpu().numpy().view(np.int8)


@pytest.mark.parametrize("n", [1, 255, 256, 257, 256 * 77 + 13, 1 << 20])
def test_quantize_and_dequantize_match_the_oracle(n):
    rng = np.random.default_rng(n)
    x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-6, 2, n)).astype(np.float32)
    x[: min(n, 300)] *= 0  # a zero block (and part of the next)
    for xdt, host in ((zdp.ZDP_F32, x), (zdp.ZDP_BF16, None)):
        if xdt == zdp.ZDP_BF16:
            xb = torch.from_numpy(x).to(torch.bfloat16)
            dx = xb.to(DEV)
            vals = xb.float().numpy()
        else:
            dx = torch.from_numpy(x).to(DEV)
            vals = x
        q = torch.empty(n, dtype=torch.int8, device=DEV)
        sc = torch.empty(-(-n // 256), dtype=torch.float32, device=DEV)
        zdp.zdp_quantize_blocks(dx, xdt, n, q, sc)
        wq, ws = oracle.quantize_blocks(vals)
        torch.cuda.synchronize()
        assert np.array_equal(_i8(q), wq), f"q n={n} xdt={xdt}"
        assert_bits_equal(sc.cpu().numpy(), ws, f"scales n={n}")
        out = torch.empty(n, dtype=torch.bfloat16, device=DEV)
        zdp.zdp_dequantize_blocks(q, sc, n, out)
        want = oracle.f32_to_bf16(oracle.dequantize_blocks(wq, ws))
        assert np.array_equal(bits_of(out), want)


def test_quantizer_near_ties_match_the_oracle():
    # Values within a few ulps of (k + 1/2) * scale, for every k and several
    # block maxima: the quotient lands on or next to a rounding tie.
    rng = np.random.default_rng(7)
    blocks = []
    for amax in [1.0, 3.0e-3, 0.7071, 123.456, 2.0 ** -60, 6.1e4]:
        a = np.float32(amax)
        sc = a / np.float32(127.0)
        centers = (np.arange(-127, 127, dtype=np.float32) + np.float32(0.5)) * sc
        vals = [centers]
        up, dn = centers.copy(), centers.copy()
        for _ in range(3):
            up = np.nextafter(up, np.float32(np.inf))
            dn = np.nextafter(dn, np.float32(-np.inf))
            vals += [up, dn]
        v = np.concatenate(vals)
        v = v[np.abs(v) <= a]
        rng.shuffle(v)
        for lo in range(0, v.size, 255):
            blk = np.zeros(256, np.float32)
            chunk = v[lo:lo + 255]
            blk[1:1 + chunk.size] = chunk
            blk[0] = a  # fixes the block maximum, hence the scale
            blocks.append(blk)
    x = np.concatenate(blocks)
    n = x.size
    q = torch.empty(n, dtype=torch.int8, device=DEV)
    sc = torch.empty(n // 256, dtype=torch.float32, device=DEV)
    zdp.zdp_quantize_blocks(torch.from_numpy(x).to(DEV), zdp.ZDP_F32, n, q, sc)
    wq, ws = oracle.quantize_blocks(x)
    torch.cuda.synchronize()
    assert_bits_equal(sc.cpu().numpy(), ws, "scales")
    got = _i8(q)
    bad = np.nonzero(got != wq)[0]
    assert bad.size == 0, f"{bad.size} codes differ, first at {bad[:4]}: {got[bad[:4]]} vs {wq[bad[:4]]}"


def _zpp_problem(P, n, seed, moments="f32"):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((P, n)) * 1e-3 * 10.0 ** rng.uniform(-1, 1, (P, 1))).astype(np.float32)
    qs = [oracle.quantize_blocks(x[r]) for r in range(P)]
    gq = np.stack([a for a, _ in qs])
    gs = np.stack([b for _, b in qs])
    S = -(-n // P)
    w = np.zeros(P * S, np.float32)
    w[:n] = rng.standard_normal(n) * 0.02
    m = np.zeros(P * S, np.float32)
    v = np.zeros(P * S, np.float32)
    m[:n] = rng.standard_normal(n) * 1e-4
    v[:n] = rng.uniform(0, 1e-6, n)
    if moments == "bf16":
        m, v = oracle.f32_to_bf16(m), oracle.f32_to_bf16(v)
    return gq, gs, w, m, v


def _to_dev(gq, gs, w, m, v, P, n, moments):
    dg = [torch.from_numpy(gq[q].view(np.uint8).copy()).to(DEV).view(torch.int8) for q in range(P)]
    ds = [torch.from_numpy(gs[q].copy()).to(DEV) for q in range(P)]
    dw = torch.from_numpy(w.copy()).to(DEV)
    if moments == "f32":
        dm, dv = torch.from_numpy(m.copy()).to(DEV), torch.from_numpy(v.copy()).to(DEV)
    else:
        dm = torch.from_numpy(m.view(np.int16).copy()).to(DEV).view(torch.bfloat16)
        dv = torch.from_numpy(v.view(np.int16).copy()).to(DEV).view(torch.bfloat16)
    nb = -(-n // 256)
    rq = [torch.zeros(n, dtype=torch.int8, device=DEV) for _ in range(P)]
    rs = [torch.zeros(nb, dtype=torch.float32, device=DEV) for _ in range(P)]
    return dg, ds, dw, dm, dv, rq, rs


@pytest.mark.parametrize("P", [1, 2, 3, 5, 8, 12, 16, 32, 64])
@pytest.mark.parametrize("moments", ["f32", "bf16"])
def test_zpp_step_matches_the_oracle(P, moments):
    for n in sorted({256 * P * 3 + 7, 40_000 + P, 256 * 64}):
        gq, gs, w, m, v = _zpp_problem(P, n, P * n, moments)
        dg, ds, dw, dm, dv, rq, rs = _to_dev(gq, gs, w, m, v, P, n, moments)
        words = torch.zeros(16, dtype=torch.uint8, device=DEV)
        a, keep = zdp.make_zpp_args(dg, ds, dw, dm, dv, rq, rs, n=n, scale=1.0 / P, t=4,
                                    d_overflow=words[0:4].view(torch.int32),
                                    d_sumsq=words[8:16].view(torch.float64), moments=moments, **HP)
        zdp.zdp_step_zpp(a)
        torch.cuda.synchronize()
        nb = gs.shape[1]
        wq, wsc = np.zeros((P, n), np.int8), np.zeros((P, nb), np.float32)
        ww, mm, vv = w.copy(), m.copy(), v.copy()
        flag, ss = oracle.step_zpp(gq, gs, ww, mm, vv, wq, wsc, n, 0, n, 1.0 / P, t=4,
                                   moments=moments, **HP)
        label = f"zpp P={P} n={n} {moments}"
        assert_state_close(dw.cpu().numpy()[:n], ww[:n], label + " master")
        if moments == "f32":
            assert_state_close(dm.cpu().numpy()[:n], mm[:n], label + " m")
            assert_state_close(dv.cpu().numpy()[:n], vv[:n], label + " v")
        else:
            assert np.array_equal(bits_of(dm)[:n], mm[:n]) and np.array_equal(bits_of(dv)[:n], vv[:n])
        for q in range(P):
            assert np.array_equal(_i8(rq[q]), wq[q]), label + f" replica {q}"
            assert_bits_equal(rs[q].cpu().numpy(), wsc[q], label + f" replica scales {q}")
        assert int(words[0:4].view(torch.int32).item()) == flag
        assert abs(float(words[8:16].view(torch.float64).item()) - ss) <= 1e-9 * ss


@pytest.mark.parametrize("P", [2, 8, 16])
@pytest.mark.parametrize("moments", ["f32", "bf16"])
@pytest.mark.parametrize("exps", [(-90, -60), (40, 70), (-90, 70)])
def test_zpp_sum_of_squares_at_extreme_scales(P, moments, exps):
    # Block scales multiplied by powers of two 2^e, e drawn from `exps`, so
    # that the squares of the reduced gradients fall below fp32's smallest
    # subnormal, above its largest value, or both within each thread's
    # share.  The P and moment types cover both accumulators of the kernel
    # (fp64 at P = 2 and at P = 8 with bf16 moments, compensated fp32 at
    # P = 8 with fp32 moments and at P = 16).
    n = 256 * 16 * P + 77
    gq, gs, w, m, v = _zpp_problem(P, n, 31 * P, moments)
    rng = np.random.default_rng(P)
    e = rng.integers(exps[0], exps[1] + 1, gs.shape)
    gs = (gs * np.exp2(e).astype(np.float32)).astype(np.float32)
    dg, ds, dw, dm, dv, rq, rs = _to_dev(gq, gs, w, m, v, P, n, moments)
    words = torch.zeros(16, dtype=torch.uint8, device=DEV)
    a, keep = zdp.make_zpp_args(dg, ds, dw, dm, dv, rq, rs, n=n, scale=1.0 / P, t=3,
                                d_overflow=words[0:4].view(torch.int32),
                                d_sumsq=words[8:16].view(torch.float64), moments=moments, **HP)
    zdp.zdp_step_zpp(a)
    torch.cuda.synchronize()
    nb = gs.shape[1]
    wq, wsc = np.zeros((P, n), np.int8), np.zeros((P, nb), np.float32)
    ww, mm, vv = w.copy(), m.copy(), v.copy()
    flag, ss = oracle.step_zpp(gq, gs, ww, mm, vv, wq, wsc, n, 0, n, 1.0 / P, t=3,
                               moments=moments, **HP)
    label = f"extreme scales P={P} {moments} 2^{exps}"
    assert flag == 0 and int(words[0:4].view(torch.int32).item()) == 0, label
    assert 0.0 < ss < np.inf and (ss < 1e-30 if exps[1] < 0 else ss > 1e20), (label, ss)
    got = float(words[8:16].view(torch.float64).item())
    assert abs(got - ss) <= 1e-9 * ss, (label, got, ss)
    assert_state_close(dw.cpu().numpy()[:n], ww[:n], label + " master")
    for q in (0, P - 1):
        assert np.array_equal(_i8(rq[q]), wq[q]), label + f" replica {q}"


@pytest.mark.parametrize("t", [200, 1000])
@pytest.mark.parametrize("moments", ["f32", "bf16"])
def test_zpp_step_in_steady_state_matches_the_oracle(t, moments):
    # From t of a few hundred on, fl(1 - b^t) is exactly 1 (at t = 1000 for
    # both betas, at t = 200 only for b1): the kernel's shortcut for that case
    # must give the oracle's bits.
    P, n = 8, 40_000
    gq, gs, w, m, v = _zpp_problem(P, n, t + 1, moments)
    dg, ds, dw, dm, dv, rq, rs = _to_dev(gq, gs, w, m, v, P, n, moments)
    a, keep = zdp.make_zpp_args(dg, ds, dw, dm, dv, rq, rs, n=n, scale=1.0 / P, t=t,
                                moments=moments, **HP)
    zdp.zdp_step_zpp(a)
    torch.cuda.synchronize()
    nb = gs.shape[1]
    wq, wsc = np.zeros((P, n), np.int8), np.zeros((P, nb), np.float32)
    ww, mm, vv = w.copy(), m.copy(), v.copy()
    oracle.step_zpp(gq, gs, ww, mm, vv, wq, wsc, n, 0, n, 1.0 / P, t=t, moments=moments, **HP)
    assert_bits_equal(dw.cpu().numpy()[:n], ww[:n], f"t={t} master")
    if moments == "f32":
        assert_bits_equal(dm.cpu().numpy()[:n], mm[:n], f"t={t} m")
        assert_bits_equal(dv.cpu().numpy()[:n], vv[:n], f"t={t} v")
    else:
        assert np.array_equal(bits_of(dm)[:n], mm[:n]) and np.array_equal(bits_of(dv)[:n], vv[:n])
    for q in range(P):
        assert np.array_equal(_i8(rq[q]), wq[q]), f"t={t} replica {q}"


def test_zpp_sub_ranges_compose_to_the_whole():
    P, n = 4, 256 * 200 + 99
    gq, gs, w, m, v = _zpp_problem(P, n, 5)
    whole = _to_dev(gq, gs, w, m, v, P, n, "f32")
    a, keep = zdp.make_zpp_args(*whole[:2], *whole[2:5], *whole[5:], n=n, scale=0.25, t=2, **HP)
    zdp.zdp_step_zpp(a)
    parts = _to_dev(gq, gs, w, m, v, P, n, "f32")
    keeps = []
    for lo, hi in ((0, 256 * 17), (256 * 17, 256 * 100), (256 * 100, n)):
        g = [x[lo:hi] for x in parts[0]]
        s_ = [x[lo // 256:] for x in parts[1]]
        b, k = zdp.make_zpp_args(g, s_, *parts[2:5], *parts[5:], n=n, scale=0.25, t=2, off=lo,
                                 length=hi - lo, **HP)
        keeps.append((b, k))
        zdp.zdp_step_zpp(b)
    torch.cuda.synchronize()
    assert_bits_equal(parts[2].cpu().numpy(), whole[2].cpu().numpy(), "master")
    for q in range(P):
        assert np.array_equal(_i8(parts[5][q]), _i8(whole[5][q]))
        assert_bits_equal(parts[6][q].cpu().numpy(), whole[6][q].cpu().numpy(), "scales")


@pytest.mark.parametrize("moments", ["f32", "bf16"])
def test_zpp_on_the_1p3b_model_sampled_blocks(moments):
    """The bench's ZeRO++ configuration (1.3B list, P = 8), both moment types,
    checked block by block against the oracle at 300 random blocks, the ends
    and every shard edge."""
    wl = workloads.gpt_1p3b()
    P, n, seed = wl.P, wl.n, 9
    S = -(-n // P)
    nb = -(-n // 256)
    gq, gs = [], []
    for q in range(P):
        g = workloads.fill_grads(torch.empty(n, dtype=torch.bfloat16, device=DEV), wl, q, 0, seed)
        qq = torch.empty(n, dtype=torch.int8, device=DEV)
        sc = torch.empty(nb, dtype=torch.float32, device=DEV)
        zdp.zdp_quantize_blocks(g, zdp.ZDP_BF16, n, qq, sc)
        del g
        gq.append(qq)
        gs.append(sc)
    st = torch.empty(3, P * S, dtype=torch.float32, device=DEV)
    workloads.fill_state(st[0], st[1], st[2], wl, seed)
    w, m, v = st[0], st[1], st[2]
    if moments == "bf16":  # the same moments held in bf16, one allocation each
        m, v = m.to(torch.bfloat16), v.to(torch.bfloat16)

    def host(t, lo, hi):
        return bits_of(t[lo:hi]).copy() if t.dtype == torch.bfloat16 else t[lo:hi].cpu().numpy().copy()

    rq = [torch.zeros(n, dtype=torch.int8, device=DEV) for _ in range(P)]
    rs = [torch.zeros(nb, dtype=torch.float32, device=DEV) for _ in range(P)]
    rng = np.random.default_rng(seed)
    blocks = sorted(set(rng.integers(0, nb, 300).tolist()) | {0, nb - 1} |
                    {(r * S) // 256 for r in range(1, P)})
    before = {}
    for b in blocks:
        lo, hi = b * 256, min(n, b * 256 + 256)
        before[b] = (host(w, lo, hi), host(m, lo, hi), host(v, lo, hi))
    a, keep = zdp.make_zpp_args(gq, gs, w, m, v, rq, rs, n=n, scale=wl.scale, t=1,
                                moments=moments, **HP)
    zdp.zdp_step_zpp(a)
    torch.cuda.synchronize()
    for b in blocks:
        lo, hi = b * 256, min(n, b * 256 + 256)
        g8 = np.stack([_i8(gq[q][lo:hi]) for q in range(P)])
        g8s = np.stack([gs[q][b:b + 1].cpu().numpy() for q in range(P)])
        ww, mm, vv = before[b]
        wq, wsc = np.zeros((P, hi - lo), np.int8), np.zeros((P, 1), np.float32)
        oracle.step_zpp(g8, g8s, ww, mm, vv, wq, wsc, n, lo, hi - lo, wl.scale, t=1, base=lo,
                        moments=moments, **HP)
        label = f"{moments} block {b}"
        assert_state_close(host(w, lo, hi), ww, label + " master")
        if moments == "f32":
            assert_state_close(host(m, lo, hi), mm, label + " m")
            assert_state_close(host(v, lo, hi), vv, label + " v")
        else:
            assert np.array_equal(host(m, lo, hi), mm), label + " m"
            assert np.array_equal(host(v, lo, hi), vv), label + " v"
        for q in (0, P - 1):
            assert np.array_equal(_i8(rq[q][lo:hi]), wq[q]), f"{label} replica {q}"
            assert rs[q][b].item() == wsc[q, 0]


@pytest.mark.parametrize("xdt", [zdp.ZDP_F32, zdp.ZDP_BF16, zdp.ZDP_FP16])
def test_quantizer_on_non_finite_blocks_matches_the_oracle(xdt):
    # A NaN makes its block's scale NaN and every code -127; an infinity makes
    # the scale infinite, its own code -127 and the others 0.
    n = 256 * 6 + 50
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    x[256 + 7] = np.nan
    x[512 + 255] = np.inf
    x[768] = -np.inf
    x[1024 + 3], x[1024 + 4] = np.nan, np.inf
    x[1536 + 49] = np.nan  # the ragged last block
    if xdt == zdp.ZDP_F32:
        dx, vals = torch.from_numpy(x).to(DEV), x
    else:
        tdt = torch.bfloat16 if xdt == zdp.ZDP_BF16 else torch.float16
        xt = torch.from_numpy(x).to(tdt)
        dx, vals = xt.to(DEV), xt.float().numpy()
    q = torch.empty(n, dtype=torch.int8, device=DEV)
    sc = torch.empty(-(-n // 256), dtype=torch.float32, device=DEV)
    zdp.zdp_quantize_blocks(dx, xdt, n, q, sc)
    wq, ws = oracle.quantize_blocks(vals)
    torch.cuda.synchronize()
    assert np.array_equal(_i8(q), wq)
    assert_bits_equal(sc.cpu().numpy(), ws, "scales")  # NaN matches NaN
    assert np.isnan(ws[1]) and ws[2] == np.inf and np.isnan(ws[4]) and np.isnan(ws[6])


@pytest.mark.parametrize("bad", [np.nan, np.inf])
@pytest.mark.parametrize("moments", ["f32", "bf16"])
def test_zpp_step_flags_a_non_finite_gradient(bad, moments):
    P, n = 8, 256 * 40 + 77
    gq, gs, w, m, v = _zpp_problem(P, n, 123, moments)
    x = (np.random.default_rng(9).standard_normal(n) * 1e-3).astype(np.float32)
    x[256 * 11 + 100] = bad
    gq[3], gs[3] = oracle.quantize_blocks(x)
    dg, ds, dw, dm, dv, rq, rs = _to_dev(gq, gs, w, m, v, P, n, moments)
    words = torch.zeros(16, dtype=torch.uint8, device=DEV)
    a, keep = zdp.make_zpp_args(dg, ds, dw, dm, dv, rq, rs, n=n, scale=1.0 / P, t=4,
                                d_overflow=words[0:4].view(torch.int32), moments=moments, **HP)
    zdp.zdp_step_zpp(a)
    torch.cuda.synchronize()
    nb = gs.shape[1]
    wq, wsc = np.zeros((P, n), np.int8), np.zeros((P, nb), np.float32)
    ww, mm, vv = w.copy(), m.copy(), v.copy()
    flag, _ = oracle.step_zpp(gq, gs, ww, mm, vv, wq, wsc, n, 0, n, 1.0 / P, t=4,
                              moments=moments, **HP)
    assert flag == 1 and int(words[0:4].view(torch.int32).item()) == 1
    assert not np.isfinite(ww[256 * 11:256 * 12]).any()
    assert_state_close(dw.cpu().numpy()[:n], ww[:n], "master")
    if moments == "f32":
        assert_state_close(dm.cpu().numpy()[:n], mm[:n], "m")
        assert_state_close(dv.cpu().numpy()[:n], vv[:n], "v")
    else:
        mb, vb = bits_of(dm)[:n], bits_of(dv)[:n]
        for got, want, name in ((mb, mm[:n], "m"), (vb, vv[:n], "v")):
            nan_w = ((want & 0x7F80) == 0x7F80) & ((want & 0x7F) != 0)
            nan_g = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
            assert np.array_equal(nan_g, nan_w) and np.array_equal(got[~nan_w], want[~nan_w]), name
    for q in range(P):
        assert np.array_equal(_i8(rq[q]), wq[q]), f"replica {q}"
        assert_bits_equal(rs[q].cpu().numpy(), wsc[q], f"replica scales {q}")
