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


def test_gpus_flag_starts_that_many_ranks():
    """``bench.py --gpus 2`` started without a torch.distributed environment
    launches two ranks itself (torch.distributed.run on 127.0.0.1, gloo on a
    machine without CUDA); rank 0 alone prints the JSON line, with n_gpus 2.
    The reference arm runs here since it needs no GPU."""
    import json
    import subprocess
    import sys

    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(os.path.dirname(bench.__file__), "bench.py"), "--gpus", "2",
                        "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
