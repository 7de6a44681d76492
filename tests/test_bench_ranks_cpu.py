"""The bench's N > 1 host logic (replicas only: no data-path collective) with two gloo
ranks on the CPU: every rank gets the slowest rank's time, and the whole-job rate counts
the units of all ranks over that time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, local_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(local_ms[rank], dist, torch.device("cpu"))
        out[rank] = (ms, bench.whole_job_rate(world, 32 * 10, ms))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    local_ms = [12.5, 20.0]
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, local_ms, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 20.0
    # 2 ranks x 32 tokens x 10 steps over 20 ms
    assert res[0][1] == pytest.approx(2 * 320 / 0.020)


def test_single_process_is_local():
    assert bench.max_over_ranks(7.0) == 7.0
    assert bench.whole_job_rate(1, 32, 1.0) == pytest.approx(32000.0)


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun only rank 0 runs and prints the reference arm."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-500:]
    assert r.stdout.strip() == ""
