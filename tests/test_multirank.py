"""bench.py's multi-rank host logic on CPU with two gloo ranks: each rank
routes its own batch (replicas), the job time is the slowest rank's, and the
reported value aggregates every rank's rows."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank  # rank 1 is slower
    ms_max = bench.max_over_ranks(ms, world)
    out[rank] = (ms_max, bench.job_throughput(8, 40, 3, world, ms_max))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms_max, value = res[rank]
        assert ms_max == 15.0
        assert value == pytest.approx(8 * 40 * 3 * world / 0.015)
