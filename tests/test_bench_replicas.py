"""Host-side logic of bench.py for more than one replica, on CPU with gloo:
every rank must end up with the slowest rank's time (the reported value is
the units all ranks processed divided by that time)."""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo")
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        q.put((rank, bench.max_over_ranks(values[rank], w)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    values = [1.5, 7.25, 3.0][:world]
    procs = [ctx.Process(target=_worker, args=(r, world, port, values, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(world))
    assert got == {r: max(values) for r in range(world)}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(4.5, 1) == 4.5
