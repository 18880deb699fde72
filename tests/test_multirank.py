"""The benchmark's multi-rank host logic on CPU with two gloo ranks: the
slowest rank's time is taken, and the whole-job throughput counts every
rank's rows (weak scaling, no collective on the data path)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        ms = [10.0, 12.5][rank]                 # rank 1 is slower
        max_ms = bench.reduce_max(ms, "cpu")
        bench.barrier()
        agg = bench.aggregate(bytes_per_step=1000, rows_per_step=4, steps=5, max_ms=max_ms,
                              world=world)
        q.put((rank, max_ms, agg))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, max_ms, agg in res:
        assert max_ms == 12.5
        # 2 ranks x 5 steps x 1000 bytes in 12.5 ms
        assert agg["gbs"] == pytest.approx(2 * 5 * 1000 / 12.5e-3 / 1e9)
        assert agg["rows_per_s"] == pytest.approx(2 * 5 * 4 / 12.5e-3)
        assert agg["ms_per_step"] == pytest.approx(12.5 / 5)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.0, "cpu") == 3.0
    agg = bench.aggregate(100, 1, 10, 1.0, 1)
    assert agg["gbs"] == pytest.approx(100 * 10 / 1e-3 / 1e9)
