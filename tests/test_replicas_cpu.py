"""The multi-GPU path of bench.py is replicas only: every rank runs its own
denoiser and the job time is the slowest rank's.  Its host-side reduction is
checked here with two gloo ranks on CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        elapsed = 100.0 + 50.0 * rank          # rank 1 is the slow one
        worst = bench.max_over_ranks(elapsed, world, torch.device("cpu"))
        value, per_rank = bench.replica_metrics(worst, 10, world)
        out[rank] = (worst, value, per_rank)
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_all_steps():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        worst, value, per_rank = res[r]
        assert worst == 150.0
        assert value == pytest.approx(150.0 / (10 * world))
        assert per_rank == pytest.approx(15.0)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1, torch.device("cpu")) == 12.5
    assert bench.replica_metrics(120.0, 10, 1) == (12.0, 12.0)
