"""The benchmark's multi-rank host logic on CPU with two gloo ranks: every rank
sees the slowest rank's timings, the whole-job throughput counts every rank's
replica, and the reference arm prints from rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    mine = [1.0 + rank, 10.0 - rank]           # rank 1 slower on the first, rank 0 on the second
    got = bench.max_over_ranks(mine, "cpu")
    dist.barrier()
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == [2.0, 10.0] and out[1] == [2.0, 10.0]


def test_job_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(1, 2e12, 1000.0) == pytest.approx(2.0)
    assert bench.job_throughput(4, 2e12, 1000.0) == pytest.approx(8.0)
    assert bench.max_over_ranks([3.0, 4.0], "cpu") == [3.0, 4.0]   # no process group: unchanged


def test_reference_arm_prints_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--gpus", "2"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
