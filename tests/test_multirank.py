"""The benchmark's multi-rank host logic on CPU: two gloo ranks (no GPU).

`bench.py --gpus N` under torchrun runs one replica of the step per GPU; the
timed region is bracketed by barriers, every rank's time is reduced to the
slowest one, and the whole-job value is N times the per-rank work over that
time.  These tests run that reduction and the value computation on two
processes over gloo."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = 10.0 + 5.0 * rank                    # rank 1 is the slow one
        worst = bench._max_over_ranks(ms, world, torch.device("cpu"))
        value = bench._job_tflops(2.0e12, world, worst)
        dist.barrier()
        out[rank] = (worst, value)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_the_whole_job_work():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]
    worst, value = res[0]
    assert worst == 15.0
    # two replicas of 2 TFLOP each in 15 ms
    assert value == pytest.approx(2 * 2.0e12 / 15e-3 / 1e12)


def test_single_rank_is_unchanged():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks(7.5, 1, torch.device("cpu")) == 7.5
    assert bench._job_tflops(1.0e12, 1, 10.0) == pytest.approx(100.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun only rank 0 times the oracle and prints; other ranks
    return at once without work."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                                      "--warmup", "0"])
    bench.main()
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    """The reference arm (the oracle on host cores) prints one JSON line with
    the keys the benchmark contract names, on rank 0."""
    import json
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    bench.main()
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == "v3_prefill"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
