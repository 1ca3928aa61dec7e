"""The benchmark's multi-rank host logic on CPU with the gloo backend (world size 2): the
timed region is the slowest rank's, the whole-job value counts every rank's steps, and the
reference arm runs on rank 0 only. No GPU: the hot path has no exchange step (replicas)."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank                        # rank 1 is the slower one
        t_max = bench.max_over_ranks(mine, world, "cpu")
        out[rank] = (t_max, bench.job_tflops(world, 1e12, 4, t_max))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as mgr:     # no fork of a multi-threaded process
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        results = dict(out)
    assert results[0][0] == results[1][0] == 15.0
    # 2 ranks x 4 steps x 1 TFLOP in 15 ms
    assert results[0][1] == pytest.approx(2 * 4 * 1.0 / 15e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_tflops(1, 2e12, 10, 20.0) == pytest.approx(10 * 2.0 / 20e-3)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    args = argparse.Namespace(steps=1, warmup=0)
    bench.run_reference(args, rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_the_contract_line():
    # the CPU oracle arm as the benchmark launches it: one JSON line with the keys and units
    # of the library's own line, warm-up raised to the minimum of three steps
    import json
    import subprocess
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOPS" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["n_gpus"] == 1 and line["steps"] == 1 and line["warmup"] >= 3
    assert line["config"]["workload"] == "contiguous_g8_t32768_n4096_k7168"
    # the same config block as the library's own arm (so the two lines describe one workload)
    import bench
    import workloads as W
    assert line["config"] == bench.headline_config(W.make_workload(bench.HEADLINE), 1)
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}

