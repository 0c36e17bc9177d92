"""The N > 1 path of bench.py on the CPU: two gloo ranks, each timing its own replica.
Both must agree on the slowest rank's time, the whole-job value counts every rank's
steps, and only rank 0 runs the reference arm."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out: str) -> None:
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        ms_local = 10.0 + 5.0 * rank  # rank 1 is the slower replica
        ms = bench.max_over_ranks(ms_local, world, "cpu")
        value = bench.whole_job_tflops(2.0e12, 4, ms, world)
        with open(f"{out}.{rank}", "w") as f:
            json.dump({"ms": ms, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_replicas_agree_on_the_slowest_rank(tmp_path):
    world, out = 2, str(tmp_path / "r")
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    res = [json.load(open(f"{out}.{r}")) for r in range(world)]
    assert res[0] == res[1]
    assert res[0]["ms"] == 15.0
    # 2 ranks x 4 steps x 2e12 flop in 15 ms
    assert res[0]["value"] == pytest.approx(2 * 4 * 2.0e12 / 15e-3 / 1e12)


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_tflops(1e12, 10, 1000.0, 1) == pytest.approx(10.0)  # 10 steps of 1e12 flop in 1 s


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    called = []
    monkeypatch.setattr(bench, "oracle_inputs", lambda w: called.append(w))
    assert bench.run_reference(None, None) is None
    assert not called
    assert capsys.readouterr().out == ""
