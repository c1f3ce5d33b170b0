"""bench.py's rank bookkeeping with two gloo ranks on the CPU.

Each rank scans its own batch (weak scaling): the seeds differ per rank, no
collective touches the data, and the reported time is the slowest rank's.
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        seconds = 0.5 + rank                       # rank 1 is the slow one
        slowest = bench.max_over_ranks(seconds)
        seed = bench.rank_seed(1, r)
        gbs = bench.aggregate_gbs(402653184, w, 10, slowest)
        out[rank] = (r, w, local, slowest, seed, gbs)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (r, w, local, slowest, seed, gbs) in res.items():
        assert (r, w, local) == (rank, 2, rank)
        assert slowest == pytest.approx(1.5)       # max over ranks, seen by every rank
        assert gbs == pytest.approx(402653184 * 2 * 10 / 1.5 / 1e9)
    assert res[0][4] == 1 and res[1][4] != res[0][4]  # rank 0 scans the named workload's own batch


def test_single_process_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.aggregate_gbs(12, 1, 1, 1e-9) == pytest.approx(12.0)
