"""The benchmark's multi-rank plumbing on CPU: two gloo ranks, each with its
own elapsed time and unit count; every rank must see the max time and the
summed units (replicas: no data-path collective is involved)."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist = bench.dist_init(world, "gloo")
    el, units = bench.aggregate(1.0 + rank, 100.0 * (rank + 1), dist, "cpu")
    results[rank] = (el, units, bench.throughput(units * 1e9, el))
    dist.destroy_process_group()


def test_two_rank_aggregate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        for r in range(world):
            el, units, gbs = results[r]
            assert el == 2.0 and units == 300.0 and gbs == 150.0


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""
