"""The benchmark's multi-rank timing path on CPU: two gloo ranks, each with
its own (simulated) step time; the job's throughput must use the slowest
rank's time and every rank's units (weak scaling, no data exchange)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, _ = bench.dist_env()
    local_seconds = 1.0 + r                      # rank 1 is slower
    slowest = bench.max_over_ranks(local_seconds, ws)
    value = bench.weak_scaling_value(10.0, ws, slowest)
    q.put((r, ws, slowest, value))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r, ws, slowest, value in out:
        assert ws == 2
        assert slowest == pytest.approx(2.0)
        assert value == pytest.approx(10.0 * 2 / 2.0)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.weak_scaling_value(8.0, 1, 2.0) == 4.0
