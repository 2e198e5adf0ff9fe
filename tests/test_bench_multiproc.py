"""The N > 1 path of bench.py on the CPU: two gloo ranks, each a replica of the
workload; the whole-job value is all units over the slowest rank's time, and
only rank 0 reports."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, _ = bench.dist_env()
    dist = bench.dist_init(w, "gloo")
    bench.barrier(dist)
    local_seconds = 1.0 + rank          # rank 1 is the slower replica
    value, slowest = bench.aggregate_replicas(10.0, local_seconds, dist)
    q.put((r, value, slowest))
    dist.destroy_process_group()


def test_two_replicas_aggregate_over_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, value, slowest in got:
        assert slowest == pytest.approx(2.0)
        assert value == pytest.approx(2 * 10.0 / 2.0)


def test_single_process_aggregate_is_identity():
    import bench
    value, slowest = bench.aggregate_replicas(6.0, 3.0, None)
    assert (value, slowest) == (2.0, 3.0)


def test_reference_arm_rank_nonzero_exits_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""
