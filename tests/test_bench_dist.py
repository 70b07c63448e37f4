"""Whole-job aggregation of bench.py over ranks (replicas, no data-path
collective): two gloo ranks on the CPU, with different local times and rows."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, rows = bench.aggregate(10.0 + 5.0 * rank, 448 * (rank + 1), world, torch.device("cpu"))
    out[rank] = (ms, rows)
    dist.destroy_process_group()


def test_aggregate_two_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == (15.0, 448 * 3)


def test_aggregate_single_rank():
    import bench
    assert bench.aggregate(3.5, 448, 1, None) == (3.5, 448)
