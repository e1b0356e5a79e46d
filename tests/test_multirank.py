"""The benchmark's N > 1 path on the CPU: two gloo ranks agree on the slowest
rank's time, the whole-job rate counts every rank's units, and under torchrun
the reference arm prints one line from rank 0 while the other rank exits 0
without work.  (One rank per GPU runs a full copy of the workload: sequences
are independent, so no collective touches the data path.)"""

from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=ws)
    try:
        bench.barrier(ws)
        ms = bench.max_over_ranks(1.0 + 3.0 * rank, ws, "cpu")  # rank 1 is the slow one
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(repr(ms))
        bench.barrier(ws)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    ws = 2
    mp.start_processes(_rank_main, args=(ws, _free_port(), str(tmp_path)), nprocs=ws, start_method="spawn")
    got = [float(open(tmp_path / f"r{r}.txt").read()) for r in range(ws)]
    assert got == [4.0, 4.0]


def test_whole_job_rate_counts_every_rank():
    assert bench.whole_job_rate(64, 1, 0.5) == pytest.approx(128000.0)
    assert bench.whole_job_rate(64, 4, 0.5) == pytest.approx(4 * 128000.0)
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5


def test_reference_arm_under_torchrun_prints_once(tmp_path):
    env = dict(os.environ, MASTER_ADDR="127.0.0.1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "insert", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=str(tmp_path))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["value"] > 0
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["cpu_baseline"]["kind"] == "oracle"
