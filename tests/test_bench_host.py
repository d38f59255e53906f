"""Host-side logic of bench.py's multi-replica path, on CPU with gloo.

With N ranks each running its own replica of the step, the job's time is the
slowest rank's and its throughput is all ranks' units over that time; the
reference arm prints from rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [12.5, 17.0][rank]
        worst = bench.max_over_ranks(ms, world, "cpu")
        q.put((rank, worst, bench.replica_throughput(1000, world, worst)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_replica_throughput_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, value in res:
        assert worst == 17.0
        assert value == pytest.approx(2 * 1000 / 0.017)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0
    assert bench.replica_throughput(500, 1, 2.0) == pytest.approx(250_000)


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True, env=env, cwd=ROOT,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env["RANK"], env["LOCAL_RANK"], env["WORLD_SIZE"] = "0", "0", "1"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True, env=env, cwd=ROOT,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0


def _bench_args(*argv):
    old = sys.argv
    sys.argv = ["bench.py", *argv]
    try:
        return bench.parse()
    finally:
        sys.argv = old


def test_profiled_traffic_only_for_the_captured_workload():
    # the committed DRAM counts belong to the full step as configured: any other
    # workload or option reports no traffic rather than another kernel's bytes
    j = json.load(open(os.path.join(ROOT, "profiles", "full_step_kernel_traffic.json")))
    assert j["workload"] == "full_step"
    got = bench.profile_traffic("bwd_tiles", _bench_args())
    assert got is None or got == float(j["kernels"]["bwd_tiles"]["dram_bytes_per_launch"])
    for argv in (["--workload", "tensornet"], ["--optimizer", "adam"], ["--batch", "1024"], ["--rows", "1000"],
                 ["--dtype", "bf16"], ["--fm"], ["--stochastic-rounding"], ["--interaction-mode", "full"]):
        assert bench.profile_traffic("bwd_tiles", _bench_args(*argv)) is None, argv
