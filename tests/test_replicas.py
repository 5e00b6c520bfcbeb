"""Replica (window-sharded) host logic of the benchmark, on CPU with two gloo ranks: the
ranks encode disjoint windows covering the global batch, and the step time is the maximum
over ranks.  The data path has no collective; these are timing-only exchanges."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wins = list(bench.rank_windows(16, rank))
    ms = bench.max_over_ranks([10.0 + rank, 3.0 - rank], dist)
    dist.destroy_process_group()
    q.put((rank, wins, ms))


def test_two_replicas_shard_windows_and_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict((r, (w, m)) for r, w, m in (q.get(timeout=120) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w0, w1 = out[0][0], out[1][0]
    assert set(w0).isdisjoint(w1) and sorted(w0 + w1) == list(range(32))
    assert out[0][1] == out[1][1] == [11.0, 3.0]


def test_single_process_has_no_reduction():
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert list(bench.rank_windows(8, 0)) == list(range(8))
