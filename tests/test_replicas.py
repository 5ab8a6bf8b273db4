"""The multi-GPU path is replicas only (every rank runs the same layers on its
own GPU, nothing exchanged on the data path): these CPU tests run its host
logic with two gloo ranks — the max over ranks of the step time, the
whole-job throughput, and the reference arm printing on rank 0 only."""
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


def _rank(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        val = bench.job_tflops(2.0e12, world, 10, ms)
        out.put((rank, ms, val))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [12.5, 20.0]  # ms of each rank's timed steps
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, ms, val in res:
        assert ms == 20.0, "every rank reports the slowest rank's time"
        # 2 ranks x 10 steps x 2 TFLOP in 20 ms = 2000 TFLOP/s
        assert val == pytest.approx(2000.0)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.job_tflops(1e12, 1, 4, 2.0) == pytest.approx(2000.0)


def test_reference_arm_prints_on_rank0_only():
    # (the oracle arm needs no GPU; a tiny layer set and one step keep it quick)
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "mnist_conv3x3_f32", "--steps", "1", "--warmup", "1"], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "", "a rank other than 0 prints nothing"
    env.update(RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "mnist_conv3x3_f32", "--steps", "1", "--warmup", "1"], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
