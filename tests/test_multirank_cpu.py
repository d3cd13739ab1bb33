"""The benchmark's multi-rank plumbing on CPU: two gloo ranks on 127.0.0.1.
On one GPU per box the path has no cross-GPU exchange, so N ranks are N
independent replicas; what must hold is the barrier and the max over ranks of
the per-rank time that rank 0 reports."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        v = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        out.put((rank, v))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_agree_on_the_max():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(world))
    assert got == {0: 15.0, 1: 15.0}


def test_single_rank_max_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
