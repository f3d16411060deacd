"""Random cases against the oracle.

Each test draws a fixed number of cases from a seeded generator and compares
every output of the library with the oracle on the same inputs.  For the
fused step the generator chooses:

- P from 1 to 64, with the compiled ranks and the generic kernel;
- n from 1 to a few hundred thousand;
- bf16 or fp16 gradients, and fp32 or bf16 moments;
- a sub-range, buckets that need not divide it, and the overflow check;
- buffers shifted off 16-byte alignment;
- injected infinities and NaNs;
- t from 1 to 1000.

The literal ring schedule, the unfused chain (reduce-scatter, AdamW on a random
slice of the shards, all-gather) and the ZeRO++ step get the same treatment:
block-aligned sub-ranges, extreme block scales and infinite scales for ZeRO++.  Master, fp32
moments, replicas, flag and quantized outputs must match bit for bit (a bf16
NaN matches any NaN, see assert_bf16_same); the sum of squares agrees within
1e-9 relative.
"""

import numpy as np
import pytest
import torch

import oracle
from harness import (HP, DeviceStep, assert_bf16_same, assert_bits_equal, bits_of,
                     random_problem)
from zero_gradient_reduce_gb300 import zdp

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")
PS = [1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 15, 16, 17, 24, 31, 32, 33, 48, 63, 64]


def _n(rng, P):
    kind = rng.integers(5)
    if kind == 0:
        return int(rng.choice([1, 2, 7, 8, 9, 15, 16, 17]))
    if kind == 1:
        return int(max(1, P + int(rng.integers(-1, 2))))
    if kind == 2:
        return int(rng.integers(1, 5000))
    return int(rng.integers(5000, max(5001, min(400_000, 12_000_000 // P))))


def _sumsq_close(got, want, label):
    if np.isfinite(want):
        assert abs(got - want) <= 1e-9 * abs(want), (label, got, want)
    else:
        assert (np.isnan(got) and np.isnan(want)) or got == want, (label, got, want)


def _step_case(rng):
    P = int(rng.choice(PS))
    n = _n(rng, P)
    gdt = oracle.FP16 if rng.random() < 0.3 else oracle.BF16
    moments = "bf16" if rng.random() < 0.3 else "f32"
    check = bool(rng.random() < 0.4)
    misalign = bool(rng.random() < 0.2)
    t = int(rng.choice([1, 2, 3, 10, 100, 1000]))
    off, length = 0, n
    if rng.random() < 0.3 and n > 2:
        off = int(rng.integers(0, n - 1))
        length = int(rng.integers(1, n - off + 1))
    bucket = int(rng.integers(max(1, length // 50), length + 1)) if rng.random() < 0.5 else 0
    gbits, w, m, v = random_problem(P, n, int(rng.integers(1 << 30)), gdt)
    inject = bool(rng.random() < 0.2)
    if inject:
        pool = [0x7C00, 0xFC00, 0x7E00] if gdt == oracle.FP16 else [0x7F80, 0xFF80, 0x7FC0]
        for _ in range(int(rng.integers(1, 3))):
            gbits[int(rng.integers(P)), int(off + rng.integers(length))] = int(rng.choice(pool))
    if moments == "bf16":
        m, v = oracle.f32_to_bf16(m), oracle.f32_to_bf16(v)
    rep = rng.integers(0, 1 << 16, (P, n), dtype=np.uint16)
    dtype = torch.float16 if gdt == oracle.FP16 else torch.bfloat16
    scale = 1.0 / (P * (65536.0 if gdt == oracle.FP16 else 1.0))
    dev = DeviceStep(P, n, dtype, misalign=misalign, moments=moments)
    dev.load(gbits, w, m, v, rep)
    dev.step(scale, t, off=off, length=length, bucket_elems=bucket, check_overflow=check)
    flag, ss = oracle.step(np.ascontiguousarray(gbits[:, off:off + length]), gdt, w, m, v, rep,
                           n, off, length, scale, t=t, check_overflow=check, moments=moments,
                           **HP)
    label = (f"P={P} n={n} off={off} len={length} bucket={bucket} gdt={gdt} "
             f"moments={moments} check={check} misalign={misalign} inject={inject} t={t}")
    got = dev.state()
    assert_bits_equal(got[0], w, f"{label} master")
    for x, y, name in zip(got[1:], (m, v), ("m", "v")):
        if moments == "f32":
            assert_bits_equal(x, y, f"{label} {name}")
        else:
            assert_bf16_same(x, y, f"{label} {name}")
    assert_bf16_same(dev.replica_bits(), rep, f"{label} replicas")
    assert int(dev.flag.item()) == flag, label
    if not (check and flag):
        _sumsq_close(float(dev.sumsq.item()), ss, label)


def _ring_case(rng):
    P = int(rng.choice([1, 2, 3, 4, 5, 8, 13, 16]))
    n = int(rng.integers(1, 3000)) if rng.random() < 0.5 else int(rng.integers(3000, 200_000))
    gbits, w, m, v = random_problem(P, n, int(rng.integers(1 << 30)), oracle.BF16)
    rep = rng.integers(0, 1 << 16, (P, n), dtype=np.uint16)
    dev = DeviceStep(P, n, torch.bfloat16, misalign=bool(rng.random() < 0.2))
    dev.load(gbits, w, m, v, rep)
    t = int(rng.choice([1, 4, 50]))
    a, keep = dev.args(1.0 / P, t)
    ws = torch.empty(zdp.zdp_step_ring_workspace_bytes(a), dtype=torch.uint8, device=DEV)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    zdp.zdp_step_ring(a)
    torch.cuda.synchronize()
    flag, ss = oracle.step(gbits, oracle.BF16, w, m, v, rep, n, 0, n, 1.0 / P, t=t, **HP)
    label = f"ring P={P} n={n} t={t}"
    for x, y, name in zip(dev.state(), (w, m, v), ("master", "m", "v")):
        assert_bits_equal(x, y, f"{label} {name}")
    assert_bf16_same(dev.replica_bits(), rep, f"{label} replicas")
    assert int(dev.flag.item()) == flag, label
    _sumsq_close(float(dev.sumsq.item()), ss, label)


def _zpp_case(rng):
    P = int(rng.choice(PS))
    n = _n(rng, P)
    moments = "bf16" if rng.random() < 0.4 else "f32"
    t = int(rng.choice([1, 3, 200, 1000]))
    nb = -(-n // 256)
    off_b = int(rng.integers(0, nb)) if rng.random() < 0.3 else 0
    off = off_b * 256
    length = min(n, int(rng.integers(off_b + 1, nb + 1)) * 256) - off
    x = (rng.standard_normal((P, n)) * 1e-3 * 10.0 ** rng.uniform(-1, 1, (P, 1))).astype(np.float32)
    if rng.random() < 0.3:  # block scales from 2^-90 to 2^70 times the usual
        x *= np.exp2(rng.integers(-90, 71, (P, 1))).astype(np.float32)
    qs = [oracle.quantize_blocks(x[r]) for r in range(P)]
    gq = np.stack([a for a, _ in qs])
    gs = np.stack([b for _, b in qs])
    inject = bool(rng.random() < 0.15)
    if inject:
        gs[int(rng.integers(P)), int(off_b + rng.integers(-(-length // 256)))] = np.float32(np.inf)
    S = -(-n // P)
    w = np.zeros(P * S, np.float32)
    m = np.zeros(P * S, np.float32)
    v = np.zeros(P * S, np.float32)
    w[:n] = rng.standard_normal(n) * 0.02
    m[:n] = rng.standard_normal(n) * 1e-4
    v[:n] = rng.uniform(0, 1e-6, n)
    if moments == "bf16":
        m, v = oracle.f32_to_bf16(m), oracle.f32_to_bf16(v)
    dg = [torch.from_numpy(gq[q, off:off + length].copy()).to(DEV) for q in range(P)]
    ds = [torch.from_numpy(gs[q, off_b:].copy()).to(DEV) for q in range(P)]
    dw = torch.from_numpy(w).to(DEV)
    if moments == "f32":
        dm, dv = torch.from_numpy(m).to(DEV), torch.from_numpy(v).to(DEV)
    else:
        dm = torch.from_numpy(m.view(np.int16).copy()).to(DEV).view(torch.bfloat16)
        dv = torch.from_numpy(v.view(np.int16).copy()).to(DEV).view(torch.bfloat16)
    rq0 = rng.integers(-128, 128, (P, n)).astype(np.int8)
    rs0 = rng.standard_normal((P, nb)).astype(np.float32)
    rq = [torch.from_numpy(rq0[q].copy()).to(DEV) for q in range(P)]
    rs = [torch.from_numpy(rs0[q].copy()).to(DEV) for q in range(P)]
    words = torch.zeros(16, dtype=torch.uint8, device=DEV)
    want_ss = bool(rng.random() < 0.7)
    a, keep = zdp.make_zpp_args(dg, ds, dw, dm, dv, rq, rs, n=n, scale=1.0 / P, t=t, off=off,
                                length=length, d_overflow=words[0:4].view(torch.int32),
                                d_sumsq=words[8:16].view(torch.float64) if want_ss else None,
                                moments=moments, **HP)
    zdp.zdp_step_zpp(a)
    torch.cuda.synchronize()
    flag, ss = oracle.step_zpp(np.ascontiguousarray(gq[:, off:off + length]),
                               np.ascontiguousarray(gs[:, off_b:]), w, m, v, rq0, rs0, n, off,
                               length, 1.0 / P, t=t, moments=moments, **HP)
    label = f"zpp P={P} n={n} off={off} len={length} moments={moments} t={t} inject={inject}"
    assert_bits_equal(dw.cpu().numpy(), w, f"{label} master")
    if moments == "f32":
        assert_bits_equal(dm.cpu().numpy(), m, f"{label} m")
        assert_bits_equal(dv.cpu().numpy(), v, f"{label} v")
    else:
        assert_bf16_same(bits_of(dm), m, f"{label} m")
        assert_bf16_same(bits_of(dv), v, f"{label} v")
    for q in range(P):
        assert np.array_equal(rq[q].cpu().numpy().view(np.int8), rq0[q]), f"{label} replica {q}"
        assert_bits_equal(rs[q].cpu().numpy(), rs0[q], f"{label} replica scales {q}")
    assert int(words[0:4].view(torch.int32).item()) == flag, label
    if want_ss:
        _sumsq_close(float(words[8:16].view(torch.float64).item()), ss, label)


def _unfused_case(rng):
    P = int(rng.choice(PS))
    n = _n(rng, P)
    S = -(-n // P)
    gdt = oracle.FP16 if rng.random() < 0.3 else oracle.BF16
    dtype = torch.float16 if gdt == oracle.FP16 else torch.bfloat16
    scale = 1.0 / (P * (65536.0 if gdt == oracle.FP16 else 1.0))
    sh = int(rng.integers(2))  # 1: every buffer one element off 16-byte alignment
    gbits, w, m, v = random_problem(P, n, int(rng.integers(1 << 30)), gdt)
    if rng.random() < 0.2:
        gbits[int(rng.integers(P)), int(rng.integers(n))] = 0x7C00 if gdt == oracle.FP16 else 0x7F80
    g_dev = [torch.from_numpy(np.concatenate([np.zeros(sh, np.uint16), gbits[q]]).view(np.int16))
             .to(DEV).view(dtype)[sh:] for q in range(P)]
    shards = torch.empty(P * S + sh, dtype=torch.float32, device=DEV)[sh:]
    words = torch.zeros(16, dtype=torch.uint8, device=DEV)
    zdp.zdp_reduce_scatter(g_dev, shards, n, P, scale, d_overflow=words[0:4].view(torch.int32),
                           d_sumsq=words[8:16].view(torch.float64))
    want, flag, ss = oracle.reduce_scatter(gbits, gdt, n, scale, want_sumsq=True)
    label = f"unfused P={P} n={n} gdt={gdt} shifted={sh}"
    assert_bits_equal(shards.cpu().numpy(), want, f"{label} shards")
    assert int(words[0:4].view(torch.int32).item()) == flag, label
    _sumsq_close(float(words[8:16].view(torch.float64).item()), ss, label)
    # AdamW on a random slice of the shards, then the all-gather of the master
    lo = int(rng.integers(0, P * S))
    count = int(rng.integers(0, P * S - lo + 1))
    t = int(rng.choice([1, 5, 1000]))
    st = torch.from_numpy(np.stack([w, m, v])).to(DEV)
    zdp.zdp_adamw_shard(st[0, lo:], st[1, lo:], st[2, lo:], shards[lo:], count, t=t, **HP)
    ww, mm, vv = w.copy(), m.copy(), v.copy()
    if count:
        ww[lo:lo + count], mm[lo:lo + count], vv[lo:lo + count] = oracle.adamw(
            w[lo:lo + count], m[lo:lo + count], v[lo:lo + count], want[lo:lo + count], t=t, **HP)
    for x, y, name in zip(st.cpu().numpy(), (ww, mm, vv), ("master", "m", "v")):
        assert_bits_equal(x, y, f"{label} adamw [{lo}, {lo + count}) {name}")
    reps = [torch.empty(n + sh, dtype=torch.bfloat16, device=DEV)[sh:] for _ in range(P)]
    zdp.zdp_all_gather(st[0], reps, n, P)
    rep_want = oracle.all_gather(ww, n, P)
    assert_bf16_same(np.stack([bits_of(r) for r in reps]), rep_want, f"{label} all-gather")


@pytest.mark.parametrize("seed", range(8))
def test_random_unfused_chains_match_the_oracle(seed):
    rng = np.random.default_rng([19, seed])
    for _ in range(10):
        _unfused_case(rng)


@pytest.mark.parametrize("seed", range(24))
def test_random_fused_steps_match_the_oracle(seed):
    rng = np.random.default_rng([11, seed])
    for _ in range(16):
        _step_case(rng)


@pytest.mark.parametrize("seed", range(4))
def test_random_ring_steps_match_the_oracle(seed):
    rng = np.random.default_rng([13, seed])
    for _ in range(10):
        _ring_case(rng)


@pytest.mark.parametrize("seed", range(12))
def test_random_zpp_steps_match_the_oracle(seed):
    rng = np.random.default_rng([17, seed])
    for _ in range(12):
        _zpp_case(rng)
