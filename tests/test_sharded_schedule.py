"""Request-sharded scheduling (Algorithm 1 over a batch split by request across
ranks): two and three gloo ranks on the CPU, each holding a shard of the
survivals (shards of different sizes), gather the batch, schedule it and keep
their own prefix lengths.  Every rank's l* must equal the single-process
schedule of the whole batch on its rows, and N and Theta_best must be the
batch's on every rank.  The scheduling step here is the oracle (the gloo path
has no GPU); on GPUs it is the library's dspark_schedule_prefix over NCCL."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

SHARDS = {2: [5, 8], 3: [7, 1, 4]}
GAMMA = 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _batch(world):
    rng = np.random.default_rng(world)
    B = sum(SHARDS[world])
    c = rng.uniform(0.3, 1.0, (B, GAMMA)).astype(np.float32)
    a = np.cumprod(c, axis=1, dtype=np.float32)
    N = np.arange(B * (GAMMA + 1) + 1, dtype=np.float64)
    return a, N / (1.0 + 0.5 * N)          # a table that saturates early: a non-trivial cut


def _oracle_schedule(a_full, sps):
    from oracle import schedule
    ell, n, th = schedule.schedule_prefix(a_full.numpy(), sps.numpy())
    return dict(ell=torch.from_numpy(np.asarray(ell)), n_sched=int(n), theta=float(th))


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from serving_draft_verify_gb300 import sharded
    a, sps = _batch(world)
    lo = sum(SHARDS[world][:rank])
    local = torch.from_numpy(a[lo:lo + SHARDS[world][rank]].copy())
    res = sharded.schedule_sharded(local, torch.from_numpy(sps), _oracle_schedule)
    out[rank] = (res["ell"].tolist(), res["n_sched"], res["theta"])
    dist.destroy_process_group()


def _check(world):
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    a, sps = _batch(world)
    from oracle import schedule
    ell, n, th = schedule.schedule_prefix(a, sps)
    lo = 0
    for r in range(world):
        got_ell, got_n, got_th = res[r]
        assert got_ell == list(ell[lo:lo + SHARDS[world][r]])
        assert got_n == n and got_th == th
        lo += SHARDS[world][r]
    assert np.any(np.asarray(ell) > 0) and np.any(np.asarray(ell) < GAMMA)   # a non-trivial cut


def test_two_ranks():
    _check(2)


def test_three_ranks_uneven_shards():
    _check(3)
