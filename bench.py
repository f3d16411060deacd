#!/usr/bin/env python
"""Benchmark of the fused ZeRO synchronisation-and-update step on one GB300.

Workload (default): the 1.3B-parameter GPT-shaped tensor list (24 layers,
d = 2048, d_ffn = 8192, vocab 50304; n = 1,311,227,904), P = 8 logical ranks
in one GPU's memory, bf16 gradients ~ N(0, sigma_T) with sigma_T
log-uniform in [1e-5, 1e-2] per tensor, fresh fp32 master/m/v.  One step is
one zdp_step over the whole model (reduce-scatter in ring order, AdamW on
every shard, bf16 cast, all-gather into all 8 replicas) plus the reset of the
overflow flag and gradient sum of squares it reports.

Prints one JSON line.  `value` is whole-job parameters per second with the
inputs resident in HBM (CUDA events on the step's stream, max over ranks);
`e2e` is the same metric through the same C ABI with the gradients copied
from pinned host memory every step and the step's flag and sum of squares
read back; `roofline` relates the fused kernel's algorithmic bytes,
(4P + 24) per parameter, to the measured HBM copy bandwidth; `cpu_baseline`
times the CPU oracle on a bounded slice of the same workload.

--impl reference times the CPU oracle alone on the same workload (a bounded
slice per step), as the reference arm.

Under torchrun with N > 1 every rank runs its own replica of the workload on
its own GPU (the step needs no exchange between GPUs: its P ranks live in
one HBM), and `value` counts all ranks' parameters over the slowest rank's
time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ZeRO step params/s and achieved HBM TB/s vs roofline (1.3B params, P=8, 1 GB300)"
HP = dict(lr=1e-4, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ("zero_gradient_reduce_gb300/csrc/zdp_kernels.cuh",
                  "zero_gradient_reduce_gb300/csrc/kernels_grad.inc",
                  "zero_gradient_reduce_gb300/csrc/zdp_internal.h")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="gpt_1p3b")
    ap.add_argument("--moments", choices=("f32", "bf16"), default="f32",
                    help="storage of the AdamW moments (bf16: 12 bytes of state per parameter)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=4)
    ap.add_argument("--e2e-bucket", type=int, default=1 << 26,
                    help="elements per rank per host->device copy bucket in the e2e leg")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-sample", type=int, default=1 << 24,
                    help="parameters per oracle step in the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-whole", action="store_true",
                    help="with --impl reference: time the oracle on whole units of the workload "
                         "instead of a bounded sample per step: one step over the whole model, "
                         "or for a streamed model its first, last and shard-straddling buckets "
                         "(minutes of CPU time and tens of GB of host memory)")
    ap.add_argument("--zpp", action="store_true",
                    help="the ZeRO++ step (int8 block-quantized gradients in, int8 replicas out) "
                         "on the workload instead of zdp_step")
    ap.add_argument("--ring-study", action="store_true",
                    help="fused step against the literal ring schedule (zdp_step_ring) for "
                         "P = 2..64: one JSON line per P")
    ap.add_argument("--sweep", action="store_true",
                    help="fp16 overflow-checked step over n = 1K..256M and P = 2..64: one "
                         "JSON line per point (cold and warm L2) instead of the benchmark line")
    ap.add_argument("--check-overflow", action="store_true",
                    help="time the overflow-checked step (skip on a non-finite reduced "
                         "gradient): one cooperative launch when the range fits one resident "
                         "wave, else two passes through a workspace")
    ap.add_argument("--overlap", action="store_true",
                    help="the ZeRO-2 streamed step: a producer stream writes each bucket's "
                         "gradients while zdp_step runs on the previous bucket on a second "
                         "stream; overlapped, producer-alone and step-alone times (default "
                         "workload of this mode: the 7B model in 256 MiB buckets)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="skip the ZeRO-2 streamed-step overlap measurement (7B model) that the "
                         "default run adds to its line")
    ap.add_argument("--unfused", action="store_true",
                    help="the three-call chain zdp_reduce_scatter -> zdp_adamw_shard -> "
                         "zdp_all_gather against the fused step, per-stage times: one JSON line")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def max_over_ranks(values, device):
    """Element-wise maximum of `values` over all ranks (identity on one rank)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(units_per_rank: int, steps: int, world: int, slowest_ms: float) -> float:
    """Units all ranks processed per second, over the slowest rank's time."""
    return world * units_per_rank * steps / (slowest_ms / 1e3)


def state_rows(length: int, device):
    """fp32 master, m and v of `length` elements as rows of one allocation,
    each row starting on a 256-byte boundary whatever P * S is (the vector
    paths want 16-byte-aligned state).  Returns (buffer, master, m, v)."""
    import torch

    row = -(-length // 64) * 64
    buf = torch.empty(3, row, dtype=torch.float32, device=device)
    return buf, buf[0, :length], buf[1, :length], buf[2, :length]


def bytes_per_param(P: int, moments: str = "f32") -> int:
    # P bf16 gradient reads + master/m/v read and written + P bf16 replica writes
    state = 12 if moments == "f32" else 8
    return 2 * P + state + state + 2 * P


def config_of(wl, bucket_elems=0, l2_flush=False, moments="f32", check_overflow=False):
    return {
        "workload": wl.name,
        "n_params": wl.n,
        "P": wl.P,
        "shard": -(-wl.n // wl.P),
        "tensors": len(wl.tensors),
        "grad_dtype": wl.grad_dtype,
        "state": ("fp32 master/m/v, bf16 replicas" if moments == "f32" else
                  "fp32 master, bf16 m/v, bf16 replicas"),
        "bucket_elems": bucket_elems,
        "check_overflow": bool(check_overflow),
        "moments": moments,
        "outputs": "overflow flag + fp64 grad sum of squares",
        "l2": ("flushed (2x L2 written) before every step; steps timed alone" if l2_flush else
               "no flush: every step streams (4P+24)n bytes, far above the 129 MB L2"),
        "parallelism": "P logical ZeRO ranks in one GPU; replicas per GPU when n_gpus > 1",
    }


GB300_L2_BYTES = 129 << 20  # a GB300's L2, about 129 MB (used where no GPU is queried)


def step_flushes_l2(wl, moments="f32", l2=GB300_L2_BYTES):
    """Whether a step of this workload moves so few bytes (under four L2
    sizes) that it is timed alone after a flush of the L2."""
    return bytes_per_param(wl.P, moments) * wl.n < 4 * l2


def fused_kernel_name(P: int, moments: str) -> str:
    """The kernel the fused step launches for P ranks and the moment type on
    the 16-byte path: the table of pick_fused_mt in csrc/kernels_grad.inc."""
    fixed = {("f32", 1), ("f32", 4), ("f32", 6), ("f32", 8), ("bf16", 1), ("bf16", 2)}
    name = "k_fused_mt" if (moments, P) in fixed else "k_fused"
    return f"{name}<P={P}, bf16 gradients, {moments} moments>"


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal


def copy_ceiling_gbs(dev, reps=10):
    """This run's device-to-device copy ceilings over 1 Gi bf16 elements, read +
    write bytes, CUDA events, best and median of `reps`: torch's b.copy_(a)
    (the way the peak in MEASURED_PEAKS.json was taken) and zdp_copy, the
    library's plain 16-byte streaming copy (the step's own access pattern)."""
    import torch

    from zero_gradient_reduce_gb300 import zdp

    a = torch.empty(1 << 30, dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    a.fill_(1.0)
    nbytes = a.numel() * a.element_size()
    stream = torch.cuda.current_stream(dev)
    out = {}
    for name, fn in (("torch_copy", lambda: b.copy_(a)),
                     ("zdp_copy", lambda: zdp.zdp_copy(b, a, nbytes, stream))):
        for _ in range(2):
            fn()
        rates = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            rates.append(2 * nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
        rates.sort()
        out[name] = (rates[-1], rates[len(rates) // 2])
    del a, b
    torch.cuda.empty_cache()
    return out


def _code_only(text: str) -> str:
    """C/C++ source without its comments and blank lines, each line stripped."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", line).strip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def kernel_source_hash() -> str:
    """sha256 prefix of the fused kernel's source files, comments excluded (a
    comment edit leaves the compiled kernel, and so its counters, as they were)."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the fused kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"zdp_fused_step_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m1 = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m2 = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    if not m1 or not m2 or m2.group(1) != kernel_source_hash():
        return None
    return float(m1.group(1))


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", self.gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [p for (t, p) in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for p in inside if num(p[2]) is not None]
        reasons = set()
        for p in inside:
            for name, val in zip(self.NAMES, p[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "power_w_max": max((num(p[3]) or 0.0) for p in inside)}


def gpu_id_for_smi(local_rank: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[local_rank]
        return str(local_rank)


# ------------------------------------------------------------------ our arm

def run_ours(args):
    import torch
    import torch.distributed as dist

    from zero_gradient_reduce_gb300 import workloads, zdp

    rank, local_rank, world = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    zdp.load()

    wl = workloads.by_name(args.workload)
    P, n = wl.P, wl.n
    S = -(-n // P)
    n_pad = P * S
    seed = args.seed + 1000 * rank
    if wl.streamed:
        run_streamed(args, wl, dev, seed, rank, world)
        return

    grads = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    for q in range(P):
        workloads.fill_grads(grads[q], wl, q, 0, seed)
    state, master, m, v = state_rows(n_pad, dev)
    workloads.fill_state(master, m, v, wl, seed)
    if args.moments == "bf16":  # the same moments, held in bf16
        # One allocation each: packed into one (2, P*S) buffer, v would start
        # 2*P*S bytes in, off the 16-byte boundary the vector path needs
        # whenever P*S is not a multiple of 8.
        m, v = m.to(torch.bfloat16), v.to(torch.bfloat16)
        master = master.clone()
        state = None
    replicas = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    words = torch.zeros(16, dtype=torch.uint8, device=dev)
    flag = words[0:4].view(torch.int32)
    sumsq = words[8:16].view(torch.float64)
    torch.cuda.synchronize()

    a, keep = zdp.make_step_args(grads, master, m, v, replicas, n=n, scale=wl.scale, t=1,
                                 bucket_elems=wl.bucket_elems, d_overflow=flag, d_sumsq=sumsq,
                                 moments=args.moments, check_overflow=args.check_overflow, **HP)
    ws = None
    if args.check_overflow:
        ws = torch.empty(zdp.zdp_step_workspace_bytes(a), dtype=torch.uint8, device=dev)
        a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    # one fused launch per bucket (the whole range when the workload has no buckets)
    launches_per_step = -(-n // wl.bucket_elems) if wl.bucket_elems else 1
    stream = torch.cuda.current_stream(dev)
    # A step that moves less than a few L2 sizes would be timed out of the L2:
    # flush it (write twice its size) before every step and time each step's
    # launches alone with events.
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = (torch.empty(2 * l2, dtype=torch.uint8, device=dev)
             if step_flushes_l2(wl, args.moments, l2) else None)
    t = 0

    def one_step(e0=None, e1=None):
        nonlocal t
        t += 1
        a.t = t
        words.zero_()
        if flush is not None:
            flush.zero_()
        if e0 is not None:
            e0.record(stream)
        zdp.zdp_step(a, stream)
        if e1 is not None:
            e1.record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_id_for_smi(local_rank))
    sampler.start()
    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    torch.cuda.nvtx.range_push("timed")  # lets a profiler restrict itself to the timed steps
    start.record(stream)
    for k in range(K):
        one_step(ev0[k], ev1[k])
    end.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    wall1 = time.time()
    if world > 1:
        dist.barrier()
    sampler.stop()
    elapsed_ms = start.elapsed_time(end)
    per_step = sorted(ev0[k].elapsed_time(ev1[k]) for k in range(K))
    kernel_ms = sum(per_step) / K
    kernel_ms_median = per_step[K // 2]
    step_flag = int(flag.item())
    if flush is not None:  # the flushes are not part of the step
        elapsed_ms = kernel_ms * K
    elapsed_ms, kernel_ms = max_over_ranks([elapsed_ms, kernel_ms], dev)
    ms_per_step = elapsed_ms / K
    value = whole_job_rate(n, K, world, elapsed_ms)

    # ---- latency floor of a step this small (timed alone after an L2 flush):
    # a minimal launch (16-byte zdp_copy) and a cold zdp_copy that moves the
    # step's own algorithmic bytes (half read, half written)
    floor = None
    if flush is not None and rank == 0:
        def cold_us(fn, reps=20):
            out = []
            for _ in range(reps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                out.append(e0.elapsed_time(e1) * 1e3)
            return sorted(out)[len(out) // 2]
        half = (bytes_per_param(P, args.moments) * n // 2 + 15) // 16 * 16
        src = torch.empty(half, dtype=torch.uint8, device=dev)
        dst = torch.empty(half, dtype=torch.uint8, device=dev)
        launch_us = cold_us(lambda: zdp.zdp_copy(dst, src, 16, stream))
        copy_us = cold_us(lambda: zdp.zdp_copy(dst, src, half, stream))
        peak_gbs = measured_peak()[0]
        floor = {"min_launch_us": launch_us, "step_bytes_copy_us": copy_us,
                 "step_bytes_at_peak_us": 2 * half / (peak_gbs * 1e3),
                 "step_us": kernel_ms_median * 1e3,
                 "step_over_copy": kernel_ms_median * 1e3 / copy_us,
                 "how": ("medians of 20, each after an L2 flush: a 16-byte zdp_copy (one "
                         "launch), and zdp_copy of the step's algorithmic bytes")}
        del src, dst

    # ---- end to end through the C ABI: gradients from pinned host memory
    e2e = None
    if not args.no_e2e and not args.check_overflow:
        e2e = run_e2e(args, wl, grads, master, m, v, replicas, words, flag, sumsq, dev, t)
        e2e["moments"] = args.moments
        slowest = max_over_ranks([e2e.get("seconds_per_step") or 0.0], dev)[0]
        if e2e.get("value") is not None:
            e2e["value"] = whole_job_rate(n, 1, world, slowest * 1e3)
        e2e.pop("seconds_per_step", None)

    copies = copy_ceiling_gbs(dev)
    copy_best, copy_median = copies["torch_copy"]

    out = None
    if rank == 0:
        peak, peak_kind = measured_peak()
        alg_bytes = bytes_per_param(P, args.moments) * n
        achieved = alg_bytes / (kernel_ms / 1e3) / 1e9
        traffic = (recorded_traffic(wl.name)
                   if args.moments == "f32" and not args.check_overflow else None)
        clocks = sampler.summary(wall0, wall1)
        out = {
            "metric": METRIC,
            "value": value,
            "unit": "params/s",
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": ms_per_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic: seeded N(0, sigma_T) bf16 gradients (sigma_T log-uniform "
                    "[1e-5, 1e-2] per tensor), master ~ N(0, 0.02), m = v = 0 at t = 1",
            "config": config_of(wl, wl.bucket_elems, flush is not None, args.moments,
                                args.check_overflow),
            "hbm_tbs": alg_bytes / (ms_per_step / 1e3) / 1e12,
            "roofline": {
                "bound": "hbm",
                "achieved": achieved,
                "peak": peak,
                "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": traffic,
                "peak_source": f"{peak_kind} HBM copy bandwidth",
                "kernel": (fused_kernel_name(P, args.moments) if not args.check_overflow else
                           "k_step_coop (one launch) or k_reduce + k_adam_gather (two passes)"),
                "algorithmic_bytes_per_launch": alg_bytes,
                "kernel_ms": kernel_ms,
                "kernel_ms_median": kernel_ms_median,
                "copy_ceiling_this_run": copy_best,
                "copy_ceiling_this_run_median": copy_median,
                "frac_of_this_run_copy": achieved / copy_best,
                "zdp_copy_this_run": copies["zdp_copy"][0],
                "zdp_copy_this_run_median": copies["zdp_copy"][1],
                "frac_of_nominal_hbm": achieved / NOMINAL_HBM_GBS,
            },
            "gpu_launches": K * launches_per_step * (2 if args.check_overflow else 1),
            "clocks": clocks,
            "overflow_flag": step_flag,
        }
        if e2e is not None:
            out["e2e"] = e2e
        if floor is not None:
            out["latency_floor"] = floor
        if args.check_overflow:
            out["metric_note"] = ("the overflow-checked step; the two-pass form moves 8 more "
                                  "bytes per parameter than the algorithmic bytes above")
        if world == 1 and not args.no_cpu_baseline and not args.check_overflow:
            out["cpu_baseline"] = cpu_baseline(args, wl, grads, master, m, v, P, n)
    # The ZeRO-2 streamed step of the 7B model, overlapped with its gradient
    # producer on a second stream (every rank runs it on its own GPU; rank 0's
    # figures are reported).  The headline buffers are freed first: the 7B
    # state and replicas take 184 GB.
    overlap = None
    if (not args.no_overlap and wl.name == workloads.gpt_1p3b().name
            and args.moments == "f32" and not args.check_overflow):
        del a, keep, grads, state, master, m, v, replicas, ws
        torch.cuda.empty_cache()
        o = overlap_measure(workloads.gpt_7b(), dev, seed, steps=3, warmup=2)
        if rank == 0:
            peak, peak_kind = measured_peak()
            gbs = lambda ms: o["step_bytes"] / (ms / 1e3) / 1e9  # noqa: E731
            overlap = {
                "workload": workloads.gpt_7b().name,
                "what": ("zdp_step per 256 MiB bucket on one stream while the producer draws the "
                         "next bucket's gradients on another (two bucket buffers)"),
                "wall_ms": o["wall_ms"], "wall_ms_each": o["wall_ms_each"],
                "producer_alone_ms": o["producer_alone_ms"],
                "step_alone_ms": o["step_alone_ms"], "sum_alone_ms": o["sum_alone_ms"],
                "hidden_ms": o["hidden_ms"],
                "step_under_contention_ms": o["step_under_contention_ms"],
                "step_alone_frac": gbs(o["step_alone_ms"]) / peak,
                "step_under_contention_frac": gbs(o["step_under_contention_ms"]) / peak,
                "peak_source": f"{peak_kind} HBM copy bandwidth", "steps": 3,
                "overflow_flag": o["overflow_flag"]}
    if out is not None and overlap is not None:
        out["streamed_overlap"] = overlap
    if out is not None and wl.name != workloads.gpt_1p3b().name:
        note = f"measured on the {wl.name} workload, not the 1.3B headline"
        out["metric_note"] = note + ("; " + out["metric_note"] if "metric_note" in out else "")
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


def run_streamed(args, wl, dev, seed, rank, world):
    """A model too large to keep every rank's gradients resident: master/m/v
    and the P replicas stay in HBM, and each step walks the model one bucket
    at a time; a bucket's P gradient slices are generated into one bucket
    buffer (outside the timed region), then zdp_step runs on that bucket with
    off/len.  The step time is the sum of the per-bucket zdp_step times
    (CUDA events on the stream around each call)."""
    import torch

    from zero_gradient_reduce_gb300 import workloads, zdp

    P, n = wl.P, wl.n
    S = -(-n // P)
    B = wl.bucket_elems
    state = [torch.empty(P * S, dtype=torch.float32, device=dev) for _ in range(3)]
    workloads.fill_state(state[0], state[1], state[2], wl, seed)
    replicas = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    bucket = [torch.empty(B, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    words = torch.zeros(16, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    bounds = [(lo, min(n, lo + B)) for lo in range(0, n, B)]
    argv = [zdp.make_step_args([b[:hi - lo] for b in bucket], state[0], state[1], state[2],
                               replicas, n=n, scale=wl.scale, t=wl.t0, off=lo, length=hi - lo,
                               d_overflow=words[0:4].view(torch.int32),
                               d_sumsq=words[8:16].view(torch.float64), **HP)
            for lo, hi in bounds]
    step_ms = []
    sampler = None
    for step in range(args.warmup + args.steps):
        if step == args.warmup:
            sampler = ClockSampler(gpu_id_for_smi(dev.index or 0))
            sampler.start()
            wall0 = time.time()
        words.zero_()
        ms = 0.0
        for (lo, hi), (a, _) in zip(bounds, argv):
            for q in range(P):
                workloads.fill_grads(bucket[q][:hi - lo], wl, q, step, seed, lo)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.t = wl.t0 + step
            e0.record(stream)
            zdp.zdp_step(a, stream)
            e1.record(stream)
            e1.synchronize()
            ms += e0.elapsed_time(e1)
        if step >= args.warmup:
            step_ms.append(ms)
    wall1 = time.time()
    sampler.stop()
    total_ms = max_over_ranks([sum(step_ms)], dev)[0]
    if rank != 0:
        return
    K = args.steps
    peak, peak_kind = measured_peak()
    alg_bytes = bytes_per_param(P) * n
    print(json.dumps({
        "metric": METRIC, "value": whole_job_rate(n, K, world, total_ms), "unit": "params/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": total_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic: seeded bf16 gradients regenerated per bucket",
        "config": dict(config_of(wl, B), l2="bucket inputs regenerated before each bucket's step"),
        "hbm_tbs": alg_bytes / (total_ms / K / 1e3) / 1e12,
        "roofline": {"bound": "hbm", "achieved": alg_bytes / (total_ms / K / 1e3) / 1e9,
                     "peak": peak, "unit": "GB/s",
                     "frac": alg_bytes / (total_ms / K / 1e3) / 1e9 / peak, "traffic": None,
                     "peak_source": f"{peak_kind} HBM copy bandwidth"},
        "gpu_launches": K * len(bounds),
        "clocks": sampler.summary(wall0, wall1),
        "metric_note": f"measured on the {wl.name} workload, not the 1.3B headline",
    }), flush=True)


def run_e2e(args, wl, grads, master, m, v, replicas, words, flag, sumsq, dev, t0):
    """End to end through the C ABI with the gradients in pinned host memory.

    Primary (`value`): the step's kernel reads the P gradient buffers straight
    from pinned host memory over the host link (GB300's host memory is mapped
    into the GPU's address space), so the step needs no staging copy; the
    flag and sum of squares are read back to the host every step.  Secondary
    (`memcpy_pipeline_value`): the gradients are copied host->device bucket by
    bucket on a copy stream, each bucket's zdp_step overlapped with the next
    bucket's copy.  Both are wall-clock times over whole steps."""
    import torch

    from zero_gradient_reduce_gb300 import zdp

    P, n = wl.P, wl.n
    try:
        host = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(P)]
    except RuntimeError as e:
        return {"value": None, "unit": "params/s", "unavailable": f"pinned host memory: {e}"[:200]}
    for q in range(P):
        host[q].copy_(grads[q])
    host_words = torch.empty(16, dtype=torch.uint8, pin_memory=True)
    main = torch.cuda.current_stream(dev)
    K = max(1, args.e2e_steps)
    t = t0

    # zero-copy: one zdp_step whose gradient pointers are the pinned host buffers
    a0, keep0 = zdp.make_step_args(host, master, m, v, replicas, n=n, scale=wl.scale, t=1,
                                   d_overflow=flag, d_sumsq=sumsq, moments=args.moments, **HP)

    def step_zero_copy():
        nonlocal t
        t += 1
        words.zero_()
        a0.t = t
        zdp.zdp_step(a0, main)
        host_words.copy_(words, non_blocking=True)
        main.synchronize()
        return int(host_words[0:4].view(torch.int32)[0])

    # memcpy pipeline
    B = max(1, args.e2e_bucket)
    bounds = [(lo, min(n, lo + B)) for lo in range(0, n, B)]
    argv = [zdp.make_step_args([g[lo:hi] for g in grads], master, m, v, replicas, n=n,
                               scale=wl.scale, t=1, off=lo, length=hi - lo, d_overflow=flag,
                               d_sumsq=sumsq, moments=args.moments, **HP) for lo, hi in bounds]
    copy = torch.cuda.Stream(dev)

    def step_memcpy():
        nonlocal t
        t += 1
        words.zero_()
        done = [torch.cuda.Event() for _ in bounds]
        copy.wait_stream(main)
        for (lo, hi), ev in zip(bounds, done):
            with torch.cuda.stream(copy):
                for q in range(P):
                    grads[q][lo:hi].copy_(host[q][lo:hi], non_blocking=True)
            ev.record(copy)
        for (a, _), ev in zip(argv, done):
            main.wait_event(ev)
            a.t = t
            zdp.zdp_step(a, main)
        host_words.copy_(words, non_blocking=True)
        main.synchronize()
        return int(host_words[0:4].view(torch.int32)[0])

    def timed(fn):
        fn()  # warm-up
        t_start = time.perf_counter()
        for _ in range(K):
            fn()
        return (time.perf_counter() - t_start) / K

    secs = timed(step_zero_copy)
    secs_memcpy = timed(step_memcpy)
    return {"value": n / secs, "unit": "params/s", "h2d_bytes_per_step": 2 * P * n,
            "d2h_bytes_per_step": 16, "steps": K,
            "method": "zdp_step reads the gradients from pinned host memory (no staging copy)",
            "gpu_launches_per_step": 1,
            "host_link_GBps": 2 * P * n / secs / 1e9,
            "memcpy_pipeline_value": n / secs_memcpy,
            "memcpy_pipeline_bucket_elems": B,
            "seconds_per_step": secs}


def _oracle_slice(P, S, n, length):
    lo = max(0, min(S - length // 2, n - length))
    return lo, min(length, n - lo)


def cpu_baseline(args, wl, grads, master, m, v, P, n):
    """The CPU oracle, as it is, on one host core, over a slice of the same
    workload straddling the boundary between rank 0's and rank 1's shards."""
    import numpy as np
    import torch

    import oracle

    S = -(-n // P)
    lo, length = _oracle_slice(P, S, n, args.cpu_sample)

    def host(t):
        x = t[lo:lo + length]
        if x.dtype == torch.float32:
            return x.cpu().numpy().copy()
        return x.view(torch.int16).cpu().numpy().view(np.uint16).copy()

    g = np.stack([host(grads[q]) for q in range(P)])
    w, mh, vh = host(master), host(m), host(v)
    rep = np.empty((P, length), np.uint16)
    oracle.build()
    steps, t0 = 0, time.perf_counter()
    while True:
        oracle.step(g, oracle.BF16, w, mh, vh, rep, n, lo, length, wl.scale, t=steps + 1,
                    base=lo, moments=args.moments, **HP)
        steps += 1
        el = time.perf_counter() - t0
        if el >= args.cpu_seconds:
            break
    return {"value": steps * length / el, "unit": "params/s", "cores": 1, "kind": "oracle",
            "host_cores": os.cpu_count(),
            "sample": f"{steps} oracle steps over params [{lo}, {lo + length}) of {wl.name} "
                      f"(P={P}, straddling the rank 0/1 shard boundary), {el:.1f} s"}


# ------------------------------------------------------------ reference arm

def run_reference(args):
    """The CPU oracle timed on the host, on the same workload and metric: each
    step is one oracle step over a bounded slice of the model."""
    import numpy as np
    import torch

    import oracle
    from zero_gradient_reduce_gb300 import workloads

    rank, _, world = dist_env()
    if rank != 0:
        return
    wl = workloads.by_name(args.workload)
    P, n = wl.P, wl.n
    S = -(-n // P)
    lo, length = _oracle_slice(P, S, n, args.cpu_sample)
    g = np.stack([workloads.fill_grads(torch.empty(length, dtype=torch.bfloat16), wl, q, 0,
                                       args.seed, lo).view(torch.int16).numpy().view(np.uint16)
                  for q in range(P)])
    gen = torch.Generator().manual_seed(workloads.key(args.seed, workloads.STREAM_MASTER))
    w = (torch.randn(length, generator=gen) * 0.02).numpy().astype(np.float32)
    m = np.zeros(length, np.float32)
    v = np.zeros(length, np.float32)
    rep = np.empty((P, length), np.uint16)
    oracle.build()
    t = 0

    if args.moments == "bf16":  # the moments held in bf16 (zeros either way)
        m, v = np.zeros(length, np.uint16), np.zeros(length, np.uint16)

    def step():
        nonlocal t
        t += 1
        oracle.step(g, oracle.BF16, w, m, v, rep, n, lo, length, wl.scale, t=t, base=lo,
                    moments=args.moments, check_overflow=args.check_overflow, **HP)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = args.steps * length / el
    sample = (f"each step: one oracle step over the {length} params [{lo}, {lo + length}) of "
              f"{wl.name} (P={P}, straddling the rank 0/1 shard boundary), single-threaded")
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "params/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        # the measured time of one step as run (one oracle step over the sample)
        "ms_per_step": el / args.steps * 1e3,
        "params_per_step": length,
        # the same per-parameter rate carried to one step over all n parameters
        "extrapolated_full_step_ms": el / args.steps * 1e3 * (n / length),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic: seeded bf16 gradients and fp32 state of the same distributions",
        "config": config_of(wl, wl.bucket_elems, step_flushes_l2(wl, args.moments),
                            args.moments, args.check_overflow),
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": 1, "kind": "oracle",
                         "host_cores": os.cpu_count(), "sample": sample},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_oracle_whole(args):
    """The CPU oracle on whole units of the workload, one host core: for a
    resident model one step over every parameter, for a streamed model
    whole buckets (the first, the last, and each one that holds a shard
    boundary), each step timed alone.  One JSON line per unit and a summary
    line.  Inputs: the workload's seeded gradients; for buckets, master/m/v
    of the workload's distributions drawn per bucket (the oracle's time does
    not depend on their values)."""
    import numpy as np
    import torch

    import oracle
    from zero_gradient_reduce_gb300 import workloads

    rank, _, world = dist_env()
    if rank != 0:
        return
    oracle.build()
    wl = workloads.by_name(args.workload)
    P, n = wl.P, wl.n
    S = -(-n // P)
    if wl.streamed:
        B = wl.bucket_elems
        bounds = [(lo, min(n, lo + B)) for lo in range(0, n, B)]
        keep = {0, len(bounds) - 1}
        keep |= {k for k, (lo, hi) in enumerate(bounds) if any(lo < r * S < hi for r in range(1, P))}
        units = [bounds[k] for k in sorted(keep)]
    else:
        units = [(0, n)]
    total_params, total_s = 0, 0.0
    for lo, hi in units:
        length = hi - lo
        g = np.empty((P, length), np.uint16)
        for q in range(P):
            t = workloads.fill_grads(torch.empty(length, dtype=torch.bfloat16), wl, q, 0,
                                     args.seed, lo)
            g[q] = t.view(torch.int16).numpy().view(np.uint16)
            del t
        rng = np.random.default_rng(workloads.key(args.seed, workloads.STREAM_MASTER, 0, 0, lo))
        w = (rng.standard_normal(length, dtype=np.float32) * np.float32(0.02))
        if wl.fresh_state:
            m = np.zeros(length, np.float32)
            v = np.zeros(length, np.float32)
        else:
            m = rng.standard_normal(length, dtype=np.float32) * np.float32(1e-4)
            v = rng.uniform(0.0, 1e-6, length).astype(np.float32)
        rep = np.empty((P, length), np.uint16)
        t0 = time.perf_counter()
        oracle.step(g, oracle.BF16, w, m, v, rep, n, lo, length, wl.scale, t=wl.t0, base=lo,
                    **HP)
        el = time.perf_counter() - t0
        total_params += length
        total_s += el
        print(json.dumps({"impl": "reference", "kind": "oracle", "workload": wl.name,
                          "unit": [lo, hi], "params": length, "seconds": el,
                          "params_per_s": length / el, "cores": 1}), flush=True)
        del g, w, m, v, rep
    print(json.dumps({
        "impl": "reference", "kind": "oracle", "workload": wl.name, "n_params": n, "P": P,
        "units": len(units), "params_timed": total_params, "seconds": total_s,
        "params_per_s": total_params / total_s, "cores": 1, "host_cores": os.cpu_count(),
        "full_step_seconds": n / (total_params / total_s),
        "what": ("one oracle step over the whole model" if not wl.streamed else
                 "whole buckets: the first, the last and each shard-straddling one"),
    }), flush=True)


def run_sweep(args):
    """GB/s of the overflow-checked step against n and P, fp16 gradients scaled
    by 2^16.  Ranges that fit one resident wave take the single-pass
    cooperative form, larger ones two passes (reduced gradients to the
    workspace, then the flag-gated AdamW + all-gather); the GB/s figure counts
    the two-pass bytes either way.  Cold: the L2 is flushed (a write of twice its
    size) before every timed step; warm: steps back to back.  Bytes per step
    are (2P + 4) n for the first pass and (4 + 24 + 2P) n for the second.

    A seeded 1 % of the runs (warm-up included) get one +inf, -inf or NaN at a
    seeded (rank, index) of the fp16 gradients, written before the run's
    start event and undone after its end event.  The flag word is cleared
    before every run; each run's flag must be 1 exactly when it was injected,
    and an injected (skipped) step does not advance t.  Each line reports the
    injected runs and whether every flag matched."""
    import numpy as np
    import torch

    from zero_gradient_reduce_gb300 import workloads, zdp

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    zdp.load()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    reps = max(3, min(args.steps, 20))
    for P in workloads.SWEEP_P:
        for n in workloads.SWEEP_N:
            wl = workloads.sweep_point(n, P)
            S = -(-n // P)
            grads = [torch.empty(n, dtype=torch.float16, device=dev) for _ in range(P)]
            for q in range(P):
                workloads.fill_grads(grads[q], wl, q, 0, args.seed)
            st = [torch.empty(P * S, dtype=torch.float32, device=dev) for _ in range(3)]
            workloads.fill_state(st[0], st[1], st[2], wl, args.seed)
            reps_buf = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
            words = torch.zeros(16, dtype=torch.uint8, device=dev)
            a, keep = zdp.make_step_args(grads, st[0], st[1], st[2], reps_buf, n=n,
                                         scale=wl.scale, t=1, check_overflow=True,
                                         d_overflow=words[0:4].view(torch.int32), **HP)
            ws = torch.empty(zdp.zdp_step_workspace_bytes(a), dtype=torch.uint8, device=dev)
            a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
            runs = args.warmup + 2 * reps
            rng = np.random.default_rng([args.seed, P, n])
            inject = rng.random(runs) < 0.01
            where = [(int(rng.integers(P)), int(rng.integers(n)),
                      int(rng.choice([0x7C00, 0xFC00, 0x7E00]))) for _ in range(runs)]
            flag = words[0:4].view(torch.int32)
            flags = torch.zeros(runs, dtype=torch.int32, device=dev)
            t = 0
            run = 0

            def one(e0=None, e1=None):
                nonlocal t, run
                k, run = run, run + 1
                flag.zero_()
                if inject[k]:
                    q, i, bits = where[k]
                    cell = grads[q].view(torch.int16)[i:i + 1]
                    saved = cell.clone()
                    cell.fill_(bits - 0x10000 if bits >= 0x8000 else bits)
                else:
                    t += 1  # an injected step is skipped and keeps t
                a.t = max(t, 1)
                if e0 is not None:
                    e0.record(stream)
                zdp.zdp_step(a, stream)
                if e1 is not None:
                    e1.record(stream)
                if inject[k]:
                    cell.copy_(saved)
                flags[k:k + 1].copy_(flag)

            for _ in range(args.warmup):
                one()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(2 * reps)]
            for k in range(reps):  # cold
                flush.zero_()
                one(*ev[k])
            for k in range(reps, 2 * reps):  # warm
                one(*ev[k])
            torch.cuda.synchronize()
            cold = sorted(e0.elapsed_time(e1) for e0, e1 in ev[:reps])[reps // 2]
            warm = sorted(e0.elapsed_time(e1) for e0, e1 in ev[reps:])[reps // 2]
            nbytes = (4 * P + 32) * n
            got = flags.cpu().numpy()
            print(json.dumps({"sweep": "fp16_checked_step", "P": P, "n": n,
                              "us_cold": cold * 1e3, "us_warm": warm * 1e3,
                              "GBps_cold": nbytes / cold / 1e6, "GBps_warm": nbytes / warm / 1e6,
                              "bytes_per_step": nbytes, "runs": runs,
                              "injected_runs": int(inject.sum()),
                              "flags_match_injections": bool(np.array_equal(got != 0, inject))}),
                  flush=True)
            del grads, st, reps_buf, ws, keep
            torch.cuda.empty_cache()


def run_ring_study(args):
    """The same step as one fused pass (zdp_step) and as the literal ring
    schedule (zdp_step_ring: P-1 reduce-scatter launches passing fp32 partial
    sums, the owner's update, P-1 all-gather launches), bf16 gradients, inputs
    resident, median of `steps` CUDA-event timings each.  busbw follows the
    nccl-tests definition for an all-reduce of the n-element bf16 gradient:
    algbw = 2n bytes / time, busbw = algbw * 2(P-1)/P."""
    import torch

    from zero_gradient_reduce_gb300 import workloads, zdp

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    zdp.load()
    stream = torch.cuda.current_stream(dev)
    for P in (2, 4, 8, 16, 64):
        n = (1 << 28) if P <= 16 else (1 << 26)
        wl = workloads.Workload(f"flat_{n}_p{P}", P=P, n=n, tensors=workloads._flat(n),
                                fresh_state=True)
        S = -(-n // P)
        grads = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
        for q in range(P):
            workloads.fill_grads(grads[q], wl, q, 0, args.seed)
        st = [torch.zeros(P * S, dtype=torch.float32, device=dev) for _ in range(3)]
        workloads.fill_state(st[0], st[1], st[2], wl, args.seed)
        reps = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
        a, keep = zdp.make_step_args(grads, st[0], st[1], st[2], reps, n=n, scale=wl.scale, t=1,
                                     **HP)
        ws = torch.empty(zdp.zdp_step_ring_workspace_bytes(a), dtype=torch.uint8, device=dev)
        res = {}
        for name, fn in (("fused", zdp.zdp_step), ("ring", zdp.zdp_step_ring)):
            if name == "ring":
                a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
            ms = []
            for k in range(args.warmup + args.steps):
                a.t = k + 1
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn(a, stream)
                e1.record(stream)
                e1.synchronize()
                if k >= args.warmup:
                    ms.append(e0.elapsed_time(e1))
            res[name] = sorted(ms)[len(ms) // 2]
        fused_b, ring_b = (4 * P + 24) * n, (14 * P + 14) * n
        algbw = lambda t: 2 * n / (t / 1e3) / 1e9
        print(json.dumps({
            "ring_study": "bf16 step", "P": P, "n": n,
            "fused_ms": res["fused"], "ring_ms": res["ring"],
            "ring_over_fused": res["ring"] / res["fused"],
            "fused_launches": 1, "ring_launches": 2 * P - 1,
            "fused_bytes": fused_b, "ring_bytes": ring_b,
            "fused_TBps": fused_b / (res["fused"] / 1e3) / 1e12,
            "ring_TBps": ring_b / (res["ring"] / 1e3) / 1e12,
            "fused_busbw_GBps": algbw(res["fused"]) * 2 * (P - 1) / P,
            "ring_busbw_GBps": algbw(res["ring"]) * 2 * (P - 1) / P,
        }), flush=True)
        del grads, st, reps, ws, keep
        torch.cuda.empty_cache()


def run_zpp(args):
    """zdp_step_zpp on the workload: each rank's bf16 gradient is block-quantized
    to int8 once (outside the timed region, as the producer would); every
    step reads the P int8 gradients and scales, updates the fp32 state and
    writes P int8 replicas and scales.  One JSON line, like the main arm."""
    import torch

    from zero_gradient_reduce_gb300 import workloads, zdp

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    zdp.load()
    wl = workloads.by_name(args.workload)
    P, n = wl.P, wl.n
    S = -(-n // P)
    nb = -(-n // zdp.ZDP_QBLOCK)
    gq, gs = [], []
    for q in range(P):
        g = workloads.fill_grads(torch.empty(n, dtype=torch.bfloat16, device=dev), wl, q, 0,
                                 args.seed)
        qq = torch.empty(n, dtype=torch.int8, device=dev)
        sc = torch.empty(nb, dtype=torch.float32, device=dev)
        zdp.zdp_quantize_blocks(g, zdp.ZDP_BF16, n, qq, sc)
        del g
        gq.append(qq)
        gs.append(sc)
    st, w, m, v = state_rows(P * S, dev)
    workloads.fill_state(w, m, v, wl, args.seed)
    if args.moments == "bf16":  # one allocation each, 16-byte aligned
        m, v = m.to(torch.bfloat16), v.to(torch.bfloat16)
    rq = [torch.empty(n, dtype=torch.int8, device=dev) for _ in range(P)]
    rs = [torch.empty(nb, dtype=torch.float32, device=dev) for _ in range(P)]
    words = torch.zeros(16, dtype=torch.uint8, device=dev)
    a, keep = zdp.make_zpp_args(gq, gs, w, m, v, rq, rs, n=n, scale=wl.scale, t=1,
                                d_overflow=words[0:4].view(torch.int32),
                                d_sumsq=words[8:16].view(torch.float64), moments=args.moments,
                                **HP)
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.warmup + args.steps)]
    sampler = ClockSampler(gpu_id_for_smi(dev.index or 0))
    sampler.start()
    wall0 = time.time()
    for k, (e0, e1) in enumerate(ev):
        a.t = k + 1
        words.zero_()
        e0.record(stream)
        zdp.zdp_step_zpp(a, stream)
        e1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    sampler.stop()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev[args.warmup:]) / args.steps
    state_b = 24 if args.moments == "f32" else 16
    bpp = 2 * P + state_b + 8 * P / zdp.ZDP_QBLOCK
    peak, peak_kind = measured_peak()
    achieved = bpp * n / (ms / 1e3) / 1e9
    print(json.dumps({
        "metric": METRIC, "value": n / (ms / 1e3), "unit": "params/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic: seeded bf16 gradients block-quantized to int8",
        "config": dict(config_of(wl, moments=args.moments),
                       state=("fp32 master/m/v" if args.moments == "f32" else
                              "fp32 master, bf16 m/v") + ", int8 replicas with block scales",
                       zpp="int8 blocks of 256, both ways"),
        "hbm_tbs": achieved / 1e3,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_kind} HBM copy bandwidth",
                     "algorithmic_bytes_per_param": bpp},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(wall0, wall1),
        "metric_note": "ZeRO++ variant of the step (quantized communication), not the headline",
    }), flush=True)


def run_unfused(args):
    """The unfused chain of the step: zdp_reduce_scatter into an fp32 shard
    buffer, zdp_adamw_shard on the whole padded range, zdp_all_gather of the
    master into the replicas.  Each stage is timed with CUDA events on the
    stream (median of `steps`), then the chain, then the fused zdp_step on
    the same buffers.  Algorithmic bytes per parameter: (2P + 4) for the
    reduce-scatter, 4 + 12 + 12 for AdamW, 4 + 2P for the all-gather:
    4P + 36 in all, against 4P + 24 fused."""
    import torch

    from zero_gradient_reduce_gb300 import workloads, zdp

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    zdp.load()
    wl = workloads.by_name(args.workload)
    P, n = wl.P, wl.n
    S = -(-n // P)
    grads = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    for q in range(P):
        workloads.fill_grads(grads[q], wl, q, 0, args.seed)
    _, *st = state_rows(P * S, dev)
    workloads.fill_state(st[0], st[1], st[2], wl, args.seed)
    shards = torch.empty(P * S, dtype=torch.float32, device=dev)
    reps = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    words = torch.zeros(16, dtype=torch.uint8, device=dev)
    flag = words[0:4].view(torch.int32)
    stream = torch.cuda.current_stream(dev)
    a, keep = zdp.make_step_args(grads, st[0], st[1], st[2], reps, n=n, scale=wl.scale, t=1,
                                 d_overflow=flag, **HP)
    t = 0

    def rs():
        zdp.zdp_reduce_scatter(grads, shards, n, P, wl.scale, d_overflow=flag, stream=stream)

    def adam():
        zdp.zdp_adamw_shard(st[0], st[1], st[2], shards, P * S, t=t, stream=stream, **HP)

    def ag():
        zdp.zdp_all_gather(st[0], reps, n, P, stream=stream)

    def chain():
        rs()
        adam()
        ag()

    def fused():
        a.t = t
        zdp.zdp_step(a, stream)

    def timed(fn):
        nonlocal t
        ms = []
        for k in range(args.warmup + args.steps):
            t += 1
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if k >= args.warmup:
                ms.append(e0.elapsed_time(e1))
        return sorted(ms)[len(ms) // 2]

    sampler = ClockSampler(gpu_id_for_smi(0))
    sampler.start()
    wall0 = time.time()
    res = {name: timed(fn) for name, fn in
           (("reduce_scatter", rs), ("adamw_shard", adam), ("all_gather", ag), ("chain", chain),
            ("fused", fused))}
    wall1 = time.time()
    sampler.stop()
    peak, peak_kind = measured_peak()
    stage_bytes = {"reduce_scatter": (2 * P + 4) * n, "adamw_shard": 28 * P * S,
                   "all_gather": (4 + 2 * P) * n, "chain": (4 * P + 36) * n,
                   "fused": (4 * P + 24) * n}
    stages = {k: {"ms": res[k], "alg_bytes": stage_bytes[k],
                  "frac_of_copy": stage_bytes[k] / (res[k] / 1e3) / 1e9 / peak} for k in res}
    print(json.dumps({
        "metric": METRIC, "value": n / (res["chain"] / 1e3), "unit": "params/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["chain"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic, as the main benchmark", "config": dict(config_of(wl), path="unfused"),
        "stages": stages, "fused_over_chain_speedup": res["chain"] / res["fused"],
        "gpu_launches": 5 * args.steps, "clocks": sampler.summary(wall0, wall1),
        "peak_source": f"{peak_kind} HBM copy bandwidth",
        "metric_note": "the unfused three-call chain, not the headline",
    }), flush=True)


def overlap_measure(wl, dev, seed, steps, warmup, stream_times=True):
    """The ZeRO-2 streamed step of `wl` (its buckets; 256 MiB per rank when it
    has none) driven by zero_gradient_reduce_gb300.streaming: the producer
    (the seeded gradient generator, standing in for the backward pass) on one
    stream, zdp_step on another, two bucket buffers.  Returns a dict of mean
    ms per step: overlapped wall time (start of the step to the last bucket's
    update), the producer alone, the steps alone (back to back on the step
    stream), and the zdp_step launches' own time inside the overlapped run
    (under contention with the producer), with the step's algorithmic bytes."""
    import torch

    from zero_gradient_reduce_gb300 import streaming, workloads, zdp

    P, n = wl.P, wl.n
    S = -(-n // P)
    B = wl.bucket_elems or (128 << 20)
    state = [torch.empty(P * S, dtype=torch.float32, device=dev) for _ in range(3)]
    workloads.fill_state(state[0], state[1], state[2], wl, seed)
    replicas = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    words = torch.zeros(16, dtype=torch.uint8, device=dev)
    ss = streaming.StreamedStep(P, n, B, state[0], state[1], state[2], replicas,
                                scale=wl.scale, d_overflow=words[0:4].view(torch.int32),
                                d_sumsq=words[8:16].view(torch.float64), device=dev, **HP)
    nb = len(ss.bounds)
    gen_step = 0

    def produce(views, lo, hi):
        for q in range(P):
            workloads.fill_bucket_grads(views[q], wl, q, gen_step, seed, lo)

    t = wl.t0
    for _ in range(warmup):
        words.zero_()
        ss.run(t, produce)
        t += 1
        gen_step += 1
    torch.cuda.synchronize()
    times = [streaming.StepTimes(nb) for _ in range(steps)]
    for k in range(steps):
        words.zero_()
        ss.run(t, produce, times[k])
        t += 1
        gen_step += 1
    torch.cuda.synchronize()
    flag = int(words[0:4].view(torch.int32).item())
    wall = sum(x.wall_ms() for x in times) / steps
    under = sum(x.step_ms() for x in times) / steps

    def alone(stream, body):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            body()  # warm-up
            for e0, e1 in ev:
                e0.record(stream)
                body()
                e1.record(stream)
        torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        return sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps

    def producer_only():
        for b, (lo, hi) in enumerate(ss.bounds):
            produce(ss.views(b), lo, hi)

    def steps_only():  # the buckets' last contents: finite gradients, same work
        for a, _ in ss.args:
            zdp.zdp_step(a, ss.stepper)

    prod_ms = alone(ss.producer, producer_only)
    step_ms = alone(ss.stepper, steps_only)
    out = {"buckets": nb, "bucket_elems": B, "wall_ms": wall,
           "wall_ms_each": [x.wall_ms() for x in times], "producer_alone_ms": prod_ms,
           "step_alone_ms": step_ms, "sum_alone_ms": prod_ms + step_ms,
           "hidden_ms": prod_ms + step_ms - wall, "step_under_contention_ms": under,
           "step_bytes": bytes_per_param(P) * n, "overflow_flag": flag,
           "producer": "seeded N(0, sigma) bf16 gradients drawn bucket by bucket "
                       "(workloads.fill_bucket_grads: one torch normal_ per rank and bucket, "
                       "per tensor slice where sigma varies by tensor), standing in for the "
                       "backward pass"}
    del ss, state, replicas
    torch.cuda.empty_cache()
    return out


def run_overlap(args):
    import torch

    from zero_gradient_reduce_gb300 import workloads, zdp

    rank, local_rank, world = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    zdp.load()
    name = args.workload if args.workload != "gpt_1p3b" else "gpt_7b"
    wl = workloads.by_name(name)
    sampler = ClockSampler(gpu_id_for_smi(local_rank))
    sampler.start()
    wall0 = time.time()
    o = overlap_measure(wl, dev, args.seed + 1000 * rank, args.steps, args.warmup)
    wall1 = time.time()
    sampler.stop()
    if rank != 0:
        return
    peak, peak_kind = measured_peak()
    n = wl.n

    def frac(ms):
        return o["step_bytes"] / (ms / 1e3) / 1e9 / peak

    print(json.dumps({
        "metric": METRIC, "value": n / (o["wall_ms"] / 1e3), "unit": "params/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": o["wall_ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic: seeded bf16 gradients drawn bucket by bucket by the producer",
        "config": dict(config_of(wl, o["bucket_elems"]),
                       l2="each bucket's gradients written by the producer just before its step",
                       streaming="two streams, two bucket buffers"),
        "overlap": dict(o, step_alone_frac=frac(o["step_alone_ms"]),
                        step_under_contention_frac=frac(o["step_under_contention_ms"]),
                        peak=peak, peak_source=f"{peak_kind} HBM copy bandwidth"),
        "gpu_launches": args.steps * o["buckets"],
        "clocks": sampler.summary(wall0, wall1),
        "metric_note": (f"the ZeRO-2 streamed step of {wl.name} overlapped with its gradient "
                        "producer: value and ms_per_step are the overlapped wall time"),
    }), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference" and args.oracle_whole:
        run_oracle_whole(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.zpp:
        run_zpp(args)
    elif args.sweep:
        run_sweep(args)
    elif args.ring_study:
        run_ring_study(args)
    elif args.unfused:
        run_unfused(args)
    elif args.overlap:
        run_overlap(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
