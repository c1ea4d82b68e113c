"""The multi-rank bench logic on CPU: two gloo ranks, one replica each.

The attention path has no exchange step (every head and query block is
independent), so N > 1 runs replicas; the only cross-rank operations are a
barrier and the max over ranks of the timed region. Those are exercised here
with the gloo backend and world size 2, without a GPU.
"""
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


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        assert (r, lr, w) == (rank, rank, world)
        dist.barrier()
        # rank 1 is the slow replica; the job time is its time
        local_seconds = 2.0 if rank == 1 else 1.0
        slowest = bench.max_over_ranks(local_seconds, dist, torch.device("cpu"))
        value = bench.job_throughput(1e12, steps=10, world=w, seconds=slowest)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{slowest} {value}")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_replica(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for rank in range(2):
        slowest, value = map(float, open(tmp_path / f"rank{rank}.txt").read().split())
        assert slowest == 2.0
        assert value == pytest.approx(1e12 * 10 * 2 / 2.0 / 1e12)   # 10 TFLOP/s for the whole job


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(2e12, steps=5, world=1, seconds=1.0) == pytest.approx(10.0)


def test_reference_arm_non_zero_ranks_do_no_work(monkeypatch):
    """Under torchrun the reference arm runs on rank 0 only; other ranks exit 0 at once."""
    from blocked_online_softmax_gb300.workloads import SMALL
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 1, 1
    assert bench.run_reference(Args(), SMALL) == 0
