"""Host logic of the multi-process bench mode, on CPU with the gloo backend.

On N GPUs the bench runs one process per GPU, each on its own full per-GPU
workload (channels are independent, so there is no collective in the data
path); the only cross-rank steps are the barrier around the timed region and
the max-over-ranks of the step time. These tests run that logic as two gloo
ranks on CPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out_path):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    w, r, lr = bench.rank_env()
    assert (w, r, lr) == (world, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks(values[rank], dist, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(f"{out_path}.{rank}", "w") as f:
        json.dump({"max": got}, f)


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    world, port = 2, _free_port()
    values = [1.25, 3.5]
    out = str(tmp_path / "res")
    mp.start_processes(_worker, args=(world, port, values, out), nprocs=world, start_method="spawn")
    for r in range(world):
        with open(f"{out}.{r}") as f:
            assert json.load(f)["max"] == max(values)


def test_job_value_is_weak_scaling():
    # every rank processes the same per-GPU units; the job's rate counts all of them
    one = bench.job_value(1, 10**9, 2.0)
    two = bench.job_value(2, 10**9, 2.0)
    assert one == pytest.approx(500.0)
    assert two == pytest.approx(2 * one)


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--gpus", "2"], env=env, capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""
