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


def _stub_measure(args, env):
    """Stands in for the GPU work of one replica: rank r takes 10 (r + 1) ms for 100 units."""
    import bench

    slow = bench.max_over_ranks(10.0 * (env.rank + 1), env.dist)
    return {"n_gpus": env.world, "rank": env.rank, "local": env.local, "steps": args.steps,
            "value": bench.aggregate_rate(env.world, 100, slow), "slow_ms": slow}


def test_gpus_flag_spawns_one_replica_per_gpu(capfd, monkeypatch):
    """`bench.py --gpus 2` with no launcher starts two replica processes (RANK = LOCAL_RANK = 0, 1) that meet
    over gloo; rank 0 alone prints the line, with the slowest rank's time."""
    import json

    import bench

    monkeypatch.delenv("WORLD_SIZE", raising=False)
    rc = bench.spawn_replicas(2, ["--gpus", "2", "--steps", "7", "--warmup", "3"], measure_fn=_stub_measure)
    assert rc == 0
    lines = [ln for ln in capfd.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["rank"] == 0 and line["local"] == 0 and line["steps"] == 7
    assert line["slow_ms"] == pytest.approx(20.0)
    assert line["value"] == pytest.approx(2 * 100 / 0.020)


def test_gpus_flag_must_match_the_launcher(monkeypatch):
    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit):
        bench.parse_args(["--gpus", "1"])
    assert bench.parse_args(["--gpus", "2"]).gpus == 2
