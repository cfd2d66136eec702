"""bench.py's multi-replica logic on CPU with two gloo ranks: the step time
reported is the max over ranks, and every rank reaches the barriers.  The
path itself has no data-path collective (replicas only)."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms = [1.25, 3.5][rank]
        got = bench.max_over_ranks(ms, world)
        # whole-job throughput: tokens of all ranks / slowest rank's time
        value = world * 16 / (got * 1e-3)
        bench.barrier(world)
        q.put((rank, got, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_max_step_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[1] for r in res] == [3.5, 3.5]
    assert res[0][2] == pytest.approx(2 * 16 / 3.5e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(2.0, 1) == 2.0
    bench.barrier(1)
