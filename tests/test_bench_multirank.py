"""The multi-rank timing logic of bench.py on CPU: world_size 2 over gloo, the job rate is all ranks' units over
the slowest rank's time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    my_ms = 10.0 * (rank + 1)  # rank 1 is the slow one
    slow = bench.max_over_ranks(my_ms, dist)
    rate = bench.aggregate_rate(world, 1000, slow)
    q.put((rank, slow, rate))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slow, rate in res:
        assert slow == pytest.approx(20.0)
        assert rate == pytest.approx(2 * 1000 / 0.020)
