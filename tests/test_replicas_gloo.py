"""The multi-GPU path of the benchmark is replicas only: every rank runs the
same product on its own GPU, the ranks meet at barriers around the timed
region, and the job's throughput is the work of all ranks over the slowest
rank's time.  These tests run that host-side logic on CPU with the gloo
backend and two ranks (no GPU involved)."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms_local = 1.0 + 0.5 * rank            # rank 1 is the slow one
        ms = bench.slowest_rank(torch, dist, torch.device("cpu"), ms_local)
        tf = bench.job_throughput(world, 2.0e9, ms)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as fh:
            fh.write(f"{ms!r} {tf!r}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_throughput(tmp_path):
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    mp.spawn(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    vals = [tuple(float(x) for x in (tmp_path / f"rank{r}.txt").read_text().split()) for r in range(world)]
    assert vals[0] == vals[1]                        # every rank reports the same figures
    ms, tf = vals[0]
    assert ms == 1.5                                 # the slowest rank's time
    assert abs(tf - world * 2.0e9 / 1.5e-3 / 1e12) < 1e-12   # all ranks' work over that time


def test_single_process_uses_its_own_time():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank(torch, None, torch.device("cpu"), 3.25) == 3.25
    assert bench.job_throughput(1, 1.0e12, 1000.0) == 1.0


def test_reference_arm_non_zero_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
