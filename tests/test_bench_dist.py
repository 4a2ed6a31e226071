"""bench.py's multi-rank path on CPU: two gloo ranks exercise the barrier, the
max-over-ranks timing, the job-wide FLOP sum and the per-rank seeds."""

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world) == bench.dist_env()[:2]
    bench.dist_barrier(world)
    t_max = bench.dist_max(10.0 + rank, world)
    f_sum = bench.dist_sum(1.5 * (rank + 1), world)
    out[rank] = (t_max, f_sum, bench.shard_seed(1001, rank))
    dist.destroy_process_group()


def test_two_rank_timing_and_aggregation():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 11.0          # slowest rank sets the time
    assert res[0][1] == res[1][1] == 1.5 + 3.0     # whole-job work
    assert res[0][2] == 1001 and res[1][2] != 1001  # rank 0 keeps the config seed


def test_single_rank_helpers_need_no_process_group():
    assert bench.dist_max(3.0, 1) == 3.0
    assert bench.dist_sum(2.0, 1) == 2.0
    bench.dist_barrier(1)
