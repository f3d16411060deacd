"""Pins of the oracle's number formats.

bf16 -> fp32 and fp16 -> fp32 are checked exhaustively (all 65,536 bit
patterns) against library conversions (torch for bf16, numpy for IEEE
binary16).  fp32 -> bf16 is checked against torch's round-to-nearest-even
conversion on special values and on random bit patterns of every class, and
against the definition itself: the result is the nearer of the two bf16
neighbours of x, ties going to the even one.
"""

import numpy as np
import torch


def _same(a, b):
    """Bitwise equal, except that any NaN matches any NaN."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    both_nan = np.isnan(a) & np.isnan(b)
    return bool(np.all(both_nan | (a.view(np.uint32) == b.view(np.uint32))))


def test_bf16_widening_exhaustive(ora):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = ora.bf16_to_f32(bits)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert _same(got, want)


def test_fp16_widening_exhaustive(ora):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = ora.f16_to_f32(bits)
    want = bits.view(np.float16).astype(np.float32)
    assert _same(got, want)
    # NaN payloads survive widening, as the IEEE widening does
    nan = np.isnan(want)
    assert np.array_equal(got[nan].view(np.uint32), want[nan].view(np.uint32))


def _torch_bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


SPECIAL = np.array([
    0.0, -0.0, 1.0, -1.0, np.inf, -np.inf,
    1.0 + 2.0 ** -8,             # exactly halfway between 1 and 1+2^-7: ties to even -> 1
    1.0 + 3 * 2.0 ** -8,         # halfway, odd lower neighbour: rounds up
    1.0 + 2.0 ** -8 + 2.0 ** -20,  # just above halfway: up
    3.3895313892515355e38,       # largest finite bf16
    3.4028234663852886e38,       # FLT_MAX rounds to +inf
    1.1754943508222875e-38,      # smallest normal
    1e-45, -1e-45,               # subnormals
    np.float32(np.pi), np.float32(-np.e), 65504.0, 1e-3, 0.02,
], dtype=np.float64).astype(np.float32)


def test_bf16_rounding_special_values(ora):
    got = ora.f32_to_bf16(SPECIAL)
    want = _torch_bf16(SPECIAL)
    assert _same(ora.bf16_to_f32(got), ora.bf16_to_f32(want))
    assert np.array_equal(got, want)  # no NaN among these
    # the hand-worked ties
    one = 0x3F80
    assert got[6] == one and got[7] == one + 2 and got[8] == one + 1


def test_bf16_rounding_random_patterns(ora):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, 2_000_000, dtype=np.uint64).astype(np.uint32)
    # force many exact ties and near-ties
    bits[:200_000] = (bits[:200_000] & 0xFFFF0000) | 0x8000
    bits[200_000:300_000] = (bits[200_000:300_000] & 0xFFFF0000) | 0x7FFF
    x = bits.view(np.float32)
    got = ora.f32_to_bf16(x)
    want = _torch_bf16(x)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all(np.isnan(ora.bf16_to_f32(got[nan])))


def test_bf16_rounding_is_nearest_even_by_definition(ora):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200_000) * 10.0 ** rng.integers(-30, 30, 200_000)).astype(np.float32)
    b = ora.f32_to_bf16(x)
    val = ora.bf16_to_f32(b).astype(np.float64)
    up = ora.bf16_to_f32((b.astype(np.uint32) + 1).astype(np.uint16)).astype(np.float64)
    dn = ora.bf16_to_f32((b.astype(np.int64) - 1).astype(np.uint16)).astype(np.float64)
    xd = x.astype(np.float64)
    err = np.abs(xd - val)
    fin = np.isfinite(val) & np.isfinite(up) & np.isfinite(dn) & (val != 0)
    assert np.all(err[fin] <= np.abs(xd - up)[fin])
    assert np.all(err[fin] <= np.abs(xd - dn)[fin])
    tie = fin & ((err == np.abs(xd - up)) | (err == np.abs(xd - dn)))
    assert np.all((b[tie] & 1) == 0)
