"""Multi-rank paths of the benchmark on CPU (gloo, world size 2): barrier, max-over-ranks
timing and rank-0-only output.  The library itself has no collective: every rank runs an
independent replica of the workload."""
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench._barrier(world)
    # each rank reports a different elapsed time; every rank must see the maximum
    t = bench._max_over_ranks(1.0 + rank, world, torch.device("cpu"))
    out[rank] = t
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_with_gloo():
    world = 2
    port = 29500 + os.getpid() % 1000
    out = mp.Manager().dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert dict(out) == {0: 2.0, 1: 2.0}


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_warmup_below_three_is_rejected():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], capture_output=True,
                       text=True, timeout=120)
    assert r.returncode != 0
