"""Host logic of the multi-GPU benchmark path, on CPU with two gloo ranks.

Every rank runs its own independent heads (weak scaling, no data-path
collective); the only collectives are the timing reductions: the step time
is the maximum over ranks and launch counts are summed.
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        shard = bench.shard_heads(2, 16, world, rank)
        maxes, sums = bench.reduce_max_sum(world, [10.0 * (rank + 1), float(rank)], [3.0 + rank],
                                           torch.device("cpu"))
        bench.barrier(world)
        out[rank] = (shard, maxes, sums)
    finally:
        dist.destroy_process_group()


def test_two_ranks_shard_and_reduce():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    # shards are disjoint batch blocks with distinct seeds, same shape
    offs = sorted(res[r][0]["batch_offset"] for r in range(world))
    assert offs == [0, 2]
    assert len({res[r][0]["seed"] for r in range(world)}) == world
    for r in range(world):
        _, maxes, sums = res[r]
        assert maxes == [20.0, 1.0]  # max over ranks, seen by every rank
        assert sums == [7.0]         # sum over ranks


def test_single_rank_reduce_is_identity():
    assert bench.reduce_max_sum(1, [1.5, 2.0], [3.0], None) == ([1.5, 2.0], [3.0])
    s = bench.shard_heads(2, 16, 1, 0)
    assert s["batch_offset"] == 0 and s["B"] == 2
