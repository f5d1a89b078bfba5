"""Host logic of the multi-GPU benchmark run, on CPU with two gloo ranks.

The decode path shards by request and has no exchange step, so several GPUs
run independent replicas: each rank times its own copy of the workload and
rank 0 reports the bytes of all ranks over the slowest rank's time.  These
checks run that reduction and the reference arm's rank handling as two
processes on the CPU.
"""
import os
import socket
import sys
import tempfile

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _aggregate_worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # rank r processed (r + 1) GB in (1 + r) / 10 seconds
        b, s = bench.aggregate(float(rank + 1) * 1e9, (1 + rank) / 10.0, world)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{b!r} {s!r}\n")
    finally:
        dist.destroy_process_group()


def test_replica_aggregate_sums_bytes_over_slowest_rank():
    world = 2
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_aggregate_worker, args=(world, _free_port(), d), nprocs=world,
                           join=True, start_method="spawn")
        for r in range(world):
            with open(os.path.join(d, f"r{r}.txt")) as f:
                b, s = (float(x) for x in f.read().split())
            assert b == 3e9          # 1 GB + 2 GB
            assert s == 0.2          # the slower rank
    # one rank: the values pass through
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(5.0, 2.0, 1) == (5.0, 2.0)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the CPU reference arm prints from rank 0 alone; the
    other ranks return at once, without drawing the workload."""
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    args = argparse.Namespace(workload="dense", steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args, world=2, rank=1) == 0


def test_dist_setup_reads_the_launcher_environment(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "4")
    monkeypatch.setenv("RANK", "3")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_setup() == (4, 3, 1)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k)
    assert bench.dist_setup() == (1, 0, 0)
