"""The N>1 path of bench.py is independent replicas: its only cross-rank
steps are the barrier and the max over ranks of the timed region.  Checked
here with two gloo ranks on the CPU."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world) == bench.dist_env()[:2]
    bench.barrier()
    got = bench.reduce_max(10.0 * (rank + 1) + 0.25)
    bench.barrier()
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((rank, got))


def test_two_rank_max_and_barrier():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 20.25, 1: 20.25}


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5) == 3.5
