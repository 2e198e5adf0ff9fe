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


def test_reference_arm_prints_the_contract_line(capsys):
    """The reference arm (the CPU oracle on a bounded sample) prints one JSON line with
    the keys the benchmark contract asks for."""
    import json

    import bench
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0", "--ref-step-s", "0.3",
                       "--workload", "ragged:127,96,512"]) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["config"]["workload"] == "ragged_residual_127x96x512"


def test_workload_names_and_bytes():
    import bench
    wl = bench.workload("mlp_gelu")
    assert bench.flops_per_step(wl) == 2.0 * 8192 * 14336 * 4096
    assert bench.algorithmic_bytes(wl) == 2.0 * (8192 * 4096 + 14336 * 4096 + 14336 + 8192 * 14336)
    rg = bench.workload("ragged:127,96,64")
    assert rg["residual"] and rg["split_k"] == "auto" and bench.needs_l2_flush(rg)
    assert not bench.needs_l2_flush(wl)
    pre = bench.workload("mlp_preact")
    assert bench.flops_per_step(pre) == bench.flops_per_step(wl)
    assert bench.algorithmic_bytes(pre) == bench.algorithmic_bytes(wl) + 2.0 * 8192 * 14336   # Z written too
    assert "Z = acc + bias" in bench.config_of(pre)["epilogue"]
