"""bench.py's replica aggregation across ranks (gloo, world size 2, CPU only).

Decode shards by sequence with no exchange, so N GPUs run N independent replicas; the
bench takes the slowest rank's step time and the sum of all ranks' KV bytes.
"""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        assert bench.dist_env() == (rank, rank, world)
        bench.barrier(world)
        ms, total = bench.aggregate(1.0 + rank, 1000 * (rank + 1), world)
        out_q.put((rank, ms, total))
    finally:
        dist.destroy_process_group()


def test_aggregate_max_time_sum_bytes():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = sorted(q.get(timeout=10) for _ in range(world))
    for _, ms, total in results:
        assert ms == pytest.approx(2.0)        # the slowest rank's time
        assert total == 3000                   # every rank's bytes


def test_single_rank_is_a_no_op():
    import bench
    assert bench.aggregate(1.5, 42, 1) == (1.5, 42)
