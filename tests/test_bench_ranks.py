"""bench.py's multi-process path (replicas): the max-over-ranks elapsed time
and the sum of units, with world_size 2 gloo ranks on the CPU."""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    el, units = bench.reduce_over_ranks(1.0 + rank, 10.0 * (rank + 1))
    bench.barrier()
    q.put((rank, el, units))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_reduce_over_ranks_gloo(world):
    import socket

    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, el, units in res:
        assert el == 2.0            # max over ranks
        assert units == 30.0        # 10 + 20


def test_single_process_passthrough():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_over_ranks(1.5, 7.0) == (1.5, 7.0)
