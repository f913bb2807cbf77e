"""The N>1 bench path on the CPU: two gloo ranks run the replica timing
aggregation (max over ranks, whole-job GB/s) that bench.py uses under torchrun."""
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
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local = [10.0 + 5.0 * rank, 3.0 - rank]  # rank 1 slower on the first, faster on the second
        got = bench.reduce_max(local)
        gbs = bench.whole_job_gbs(2_000_000_000, 4, world, got[0])
        q.put((rank, got, gbs))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, gbs in res:
        assert got == [15.0, 3.0]
        # 2 replicas x 4 rounds x 2 GB in 15 ms
        assert gbs == pytest.approx(2 * 4 * 2.0 / 0.015)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max([1.5, 2.5]) == [1.5, 2.5]
    assert bench.whole_job_gbs(10**9, 10, 1, 1000.0) == pytest.approx(10.0)
