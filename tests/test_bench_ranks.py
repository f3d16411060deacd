"""The benchmark's multi-GPU bookkeeping on CPU: two gloo ranks (one process
each, rendezvous on 127.0.0.1) take the element-wise maximum of their timings
and report the whole job's rate over the slowest rank; the reference arm
prints from rank 0 only."""

import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        got = bench.max_over_ranks([10.0 + rank, 5.0 - rank], "cpu")
        out[rank] = got + [bench.whole_job_rate(1000, 4, world, got[0])]
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        ps = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in ps:
            p.start()
        for p in ps:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(2):
        assert res[r][:2] == [11.0, 5.0]
        # 2 ranks x 1000 units x 4 steps over 11 ms
        assert res[r][2] == pytest.approx(2 * 1000 * 4 / 0.011)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([3.0, 4.0], "cpu") == [3.0, 4.0]
    assert bench.whole_job_rate(10, 2, 1, 1000.0) == pytest.approx(20.0)


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", "--cpu-sample", "4096"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_line():
    import json

    env = dict(os.environ, RANK="0", LOCAL_RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1", "--cpu-sample", "65536"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "params/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_headline_profile_matches_the_kernel_sources():
    # bench.py reports the committed ncu traffic only while the kernel sources
    # hash to the value recorded beside it; a kernel change without a new
    # capture would silently turn `traffic` into null.
    sys.path.insert(0, ROOT)
    import bench

    traffic = bench.recorded_traffic("gpt_1.3B_p8")
    assert traffic is not None, "kernel sources changed since profiles/ was captured"
    alg = 56 * 1_311_227_904
    assert 0.99 * alg < traffic < 1.01 * alg


def test_kernel_label_follows_the_fused_dispatch_table():
    # The benchmark line names the fused kernel from its own copy of the
    # table in pick_fused_mt (csrc/kernels_grad.inc); the two must agree.
    import re

    sys.path.insert(0, ROOT)
    import bench

    src = open(os.path.join(ROOT, "zero_gradient_reduce_gb300", "csrc", "kernels_grad.inc")).read()
    body = src[src.index("const void* pick_fused_mt(int P, int mt) {"):]
    body = body[:body.index("\n}\n")]
    table = set()
    for P, mt in re.findall(r"case (\d+): return reinterpret_cast<const void\*>\(&k_fused_mt<\d+, ZDP_GT, ZDP_MOMENTS_(F32|BF16)", body):
        table.add(("f32" if mt == "F32" else "bf16", int(P)))
    assert table, "no k_fused_mt cases found"
    for moments in ("f32", "bf16"):
        for P in range(1, 65):
            named = bench.fused_kernel_name(P, moments).startswith("k_fused_mt<")
            assert named == ((moments, P) in table), (moments, P)


def test_source_hash_ignores_comments_but_not_code():
    sys.path.insert(0, ROOT)
    import bench

    code = "int f(int x) {  // doubles\n  return 2 * x; /* two\n lines */\n}\n"
    assert bench._code_only(code) == bench._code_only(
        "int f(int x) {\n\n  return 2 * x;   // another note\n}\n")
    assert bench._code_only(code) != bench._code_only(code.replace("2 * x", "3 * x"))


def test_flat_slice_workloads_by_name():
    from zero_gradient_reduce_gb300 import workloads

    for P in (1, 2, 8, 64):
        wl = workloads.by_name(f"flat_p{P}_32m")
        assert wl.P == P and wl.n == 32 * 2**20 and wl.fresh_state
    assert workloads.by_name("flat_p8_32m").name == workloads.flat_p8_32m().name
    with pytest.raises(KeyError):
        workloads.by_name("flat_px_32m")


def test_state_rows_start_on_256_byte_boundaries():
    """The bench's master, m and v rows stay 16-byte aligned (the vector paths
    need it) whatever P * S is, e.g. P = 3 on the 32M slice."""
    import bench

    for length in (1, 7, 33554433, 33554436):
        buf, w, m, v = bench.state_rows(length, "cpu")
        assert w.numel() == m.numel() == v.numel() == length
        base = buf.data_ptr()
        for row in (w, m, v):
            assert (row.data_ptr() - base) % 256 == 0
            assert row.is_contiguous()
