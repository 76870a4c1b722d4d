"""The multi-GPU path is replicas only (one independent decode per rank, no
collective in the data path); bench.py's only exchange is the max over ranks
of the step timings. Checked here with world_size 2 over gloo on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r saw step times (10 + r, 30 - r): the job's are the maxima
        out[rank] = bench.max_over_ranks([10.0 + rank, 30.0 - rank], world, "cpu")
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_world2_gloo():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        got = dict(out)
    assert got[0] == [11.0, 30.0] and got[1] == [11.0, 30.0]


def test_max_over_ranks_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([3.5, 7], 1) == [3.5, 7.0]


def test_reference_arm_runs_on_rank0_only():
    import argparse
    import bench
    assert bench.run_reference(argparse.Namespace(workload="tiny_two_level"), rank=1) is None
