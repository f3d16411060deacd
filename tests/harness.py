"""Helpers shared by the tests: moving seeded inputs between host and device,
running the library through its C ABI, and the parity comparisons.

Tolerances (the step's target): reduced gradients and the overflow flag
bit-exact; fp32 master, m and v within 1e-6 relative (absolute floor 1e-30
for zeros); bf16 replicas within 1 bf16 ulp; NaN matches NaN.  The library
evaluates the same IEEE operations in the same order as the oracle, so in
practice every comparison below is exact; the tests still state and enforce
the tolerance, and report the largest deviation they saw.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from zero_gradient_reduce_gb300 import workloads, zdp

STATE_RTOL = 1e-6
STATE_ATOL_FLOOR = 1e-30
REPLICA_ULP = 1

HP = dict(lr=1e-4, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)


def bits_of(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16/fp16 tensor, on the host."""
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def tensor_from_bits(bits: np.ndarray, dtype, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(dtype)


def gdt_of(dtype) -> int:
    return zdp.ZDP_FP16 if dtype == torch.float16 else zdp.ZDP_BF16


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if got.dtype == np.float32:
        nan = np.isnan(got) & np.isnan(want)
        bad = ~nan & (got.view(np.uint32) != want.view(np.uint32))
    else:
        bad = got != want
    if bad.any():
        i = int(np.flatnonzero(bad.ravel())[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} differ; first at {i}: "
                             f"got {got.ravel()[i]!r} want {want.ravel()[i]!r}")


def assert_state_close(got: np.ndarray, want: np.ndarray, what: str) -> float:
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape
    nan_g, nan_w = np.isnan(got), np.isnan(want)
    assert np.array_equal(nan_g, nan_w), f"{what}: NaN positions differ"
    ok = ~nan_w
    g64, w64 = got[ok].astype(np.float64), want[ok].astype(np.float64)
    inf = np.isinf(w64) | np.isinf(g64)
    assert np.array_equal(g64[inf], w64[inf]), f"{what}: infinities differ"
    g64, w64 = g64[~inf], w64[~inf]
    rel = np.abs(g64 - w64) / np.maximum(np.abs(w64), STATE_ATOL_FLOOR)
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= STATE_RTOL, f"{what}: max relative error {worst:.3g} > {STATE_RTOL}"
    return worst


def _ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def assert_bf16_close(got: np.ndarray, want: np.ndarray, what: str) -> int:
    got = np.asarray(got, np.uint16)
    want = np.asarray(want, np.uint16)
    assert got.shape == want.shape
    nan_g = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    nan_w = ((want & 0x7F80) == 0x7F80) & ((want & 0x7F) != 0)
    assert np.array_equal(nan_g, nan_w), f"{what}: NaN positions differ"
    d = np.abs(_ordered(got[~nan_w]) - _ordered(want[~nan_w]))
    worst = int(d.max()) if d.size else 0
    assert worst <= REPLICA_ULP, f"{what}: {worst} bf16 ulp apart"
    return worst


def assert_bf16_same(got: np.ndarray, want: np.ndarray, what: str):
    """bf16 bit patterns equal, except that a NaN matches any NaN: IEEE 754
    leaves the sign and payload of a NaN made by an invalid operation to the
    implementation (the GPU's conversion writes 0x7FFF, the oracle keeps the
    sign of its host's NaN with 0x7FC0)."""
    got = np.asarray(got, np.uint16)
    want = np.asarray(want, np.uint16)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    nan_g = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    nan_w = ((want & 0x7F80) == 0x7F80) & ((want & 0x7F) != 0)
    assert np.array_equal(nan_g, nan_w), f"{what}: NaN positions differ"
    bad = (got != want) & ~nan_w
    if bad.any():
        i = int(np.flatnonzero(bad.ravel())[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} differ; first at {i}: "
                             f"got {got.ravel()[i]:#06x} want {want.ravel()[i]:#06x}")


class DeviceStep:
    """Device buffers of one step problem: P gradients (bf16/fp16), fp32
    master/m/v of n_pad elements, P bf16 replicas, flag and sum of squares."""

    def __init__(self, P: int, n: int, gdtype=torch.bfloat16, device="cuda", misalign=False,
                 moments="f32"):
        self.P, self.n = P, n
        self.S = -(-n // P)
        self.n_pad = P * self.S
        self.device = device
        self.moments = moments
        extra = 1 if misalign else 0
        self._g = [torch.zeros(n + extra, dtype=gdtype, device=device) for _ in range(P)]
        self._r = [torch.zeros(n + extra, dtype=torch.bfloat16, device=device) for _ in range(P)]
        self._st = torch.zeros(3, self.n_pad + 4 * extra, dtype=torch.float32, device=device)
        self.grads = [g[extra:] for g in self._g]
        self.replicas = [r[extra:] for r in self._r]
        self.master = self._st[0, extra:extra + self.n_pad]
        if moments == "f32":
            self.m = self._st[1, extra:extra + self.n_pad]
            self.v = self._st[2, extra:extra + self.n_pad]
        else:  # bf16 moments, separate buffers
            self._mv = torch.zeros(2, self.n_pad + 8 * extra, dtype=torch.bfloat16, device=device)
            self.m = self._mv[0, extra:extra + self.n_pad]
            self.v = self._mv[1, extra:extra + self.n_pad]
        self.flag = torch.zeros(1, dtype=torch.int32, device=device)
        self.sumsq = torch.zeros(1, dtype=torch.float64, device=device)

    def load(self, gbits: np.ndarray, w, m, v, rep_bits=None):
        for q in range(self.P):
            self.grads[q].copy_(tensor_from_bits(gbits[q, :self.n], self.grads[q].dtype, "cpu"))
        self.master.copy_(torch.from_numpy(np.asarray(w, np.float32)))
        if self.moments == "f32":
            self.m.copy_(torch.from_numpy(np.asarray(m, np.float32)))
            self.v.copy_(torch.from_numpy(np.asarray(v, np.float32)))
        else:  # m, v given as bf16 bit patterns
            self.m.copy_(tensor_from_bits(np.asarray(m, np.uint16), torch.bfloat16, "cpu"))
            self.v.copy_(tensor_from_bits(np.asarray(v, np.uint16), torch.bfloat16, "cpu"))
        if rep_bits is not None:
            for q in range(self.P):
                self.replicas[q].copy_(tensor_from_bits(rep_bits[q], torch.bfloat16, "cpu"))

    def state(self):
        if self.moments == "f32":
            return (self.master.cpu().numpy(), self.m.cpu().numpy(), self.v.cpu().numpy())
        return (self.master.cpu().numpy(), bits_of(self.m), bits_of(self.v))

    def replica_bits(self) -> np.ndarray:
        return np.stack([bits_of(r) for r in self.replicas])

    def args(self, scale, t, off=0, length=None, bucket_elems=0, check_overflow=False,
             workspace=None, with_flag=True, with_sumsq=True, **hp):
        hp = {**HP, **hp}
        length = self.n - off if length is None else length
        grads = [g[off:off + length] if length > 0 else g for g in self.grads]
        a, keep = zdp.make_step_args(
            grads, self.master, self.m, self.v, self.replicas, n=self.n, scale=scale, t=t,
            off=off, length=length, bucket_elems=bucket_elems, check_overflow=check_overflow,
            d_overflow=self.flag if with_flag else None,
            d_sumsq=self.sumsq if with_sumsq else None, moments=self.moments, **hp)
        if check_overflow:
            nbytes = zdp.zdp_step_workspace_bytes(a)
            if workspace is None:
                workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            a.workspace = workspace.data_ptr()
            a.workspace_bytes = workspace.numel()
        return a, (keep, workspace)

    def step(self, scale, t, **kw):
        a, keep = self.args(scale, t, **kw)
        zdp.zdp_step(a)
        torch.cuda.synchronize()
        return keep


def random_problem(P, n, seed, gdt=oracle.BF16, fresh=False, grad_scale=1e-3):
    """Seeded host inputs of the parity cases: gradients ~ N(0, grad_scale)
    (times 2^16 for fp16), master ~ N(0, 0.02), m ~ N(0, 1e-4), v ~ U[0, 1e-6]."""
    rng = np.random.default_rng(seed)
    S = -(-n // P)
    g = rng.standard_normal((P, n)).astype(np.float32) * np.float32(grad_scale)
    if gdt == oracle.FP16:
        gbits = (g * np.float32(65536.0)).astype(np.float16).view(np.uint16)
    else:
        gbits = torch.from_numpy(g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    w = np.zeros(P * S, np.float32)
    m = np.zeros(P * S, np.float32)
    v = np.zeros(P * S, np.float32)
    w[:n] = rng.standard_normal(n) * 0.02
    if not fresh:
        m[:n] = rng.standard_normal(n) * 1e-4
        v[:n] = rng.uniform(0, 1e-6, n)
    return np.ascontiguousarray(gbits), w, m, v


class SampledProducer:
    """produce() callback: writes the seeded gradients of a bucket and keeps
    the values at the sampled indices that fall in it (on the producer
    stream, right after writing them)."""

    def __init__(self, wl, seed, idx, P, fill=workloads.fill_grads):
        self.wl, self.seed, self.P, self.fill = wl, seed, P, fill
        self.idx = idx
        self.gs = torch.zeros((P, idx.size), dtype=torch.int16, device="cuda")
        self.step = 0

    def prepare(self, bounds):
        self.sel = []
        for lo, hi in bounds:
            k = np.nonzero((self.idx >= lo) & (self.idx < hi))[0]
            self.sel.append((torch.from_numpy(k).cuda(),
                             torch.from_numpy(self.idx[k] - lo).cuda()))
        torch.cuda.synchronize()
        self.bounds = bounds

    def __call__(self, views, lo, hi):
        b = self.bounds.index((lo, hi))
        pos, local = self.sel[b]
        for q in range(self.P):
            self.fill(views[q], self.wl, q, self.step, self.seed, lo)
            self.gs[q].index_copy_(0, pos, views[q].view(torch.int16).index_select(0, local))

    def host_values(self):
        return self.gs.cpu().numpy().view(np.uint16)
