"""The multi-rank path of bench.py on CPU: two gloo ranks on 127.0.0.1.

bench.py runs one replica of the workload per GPU rank (the (sequence, head)
chains are independent, so nothing is exchanged on the data path).  What the
ranks share is the timing: the job's time is the slowest rank's, and the
reported rate counts every rank's tokens.  These tests run that reduction and
the rank gating of the reference arm with the gloo backend, no GPU involved.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        rate = bench.whole_job_rate(1000, world, 4, m)
        out[rank] = (m, rate)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_every_rank():
    world, port = 2, _free_port()
    times = [12.5, 20.0]          # ms for 4 steps on each rank
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        m, rate = res[r]
        assert m == 20.0
        # 2 ranks x 4 steps x 1000 tokens in 20 ms
        assert rate == pytest.approx(2 * 4 * 1000 / 0.020)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(7.0, 1, torch.device("cpu")) == 7.0
    assert bench.whole_job_rate(500, 1, 2, 10.0) == pytest.approx(500 * 2 / 0.010)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(None, bench.workload("tiny")) is None
    assert capsys.readouterr().out == ""


def test_backward_reference_arm_prints_one_oracle_line(monkeypatch, capsys):
    import json
    import types

    monkeypatch.delenv("RANK", raising=False)
    args = types.SimpleNamespace(steps=1, warmup=0, gpus=1)
    bench.run_bwd_reference(args, bench.workload("tiny"))
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["metric"] == bench.BWD_METRIC
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] == line["cpu_baseline"]["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["pass"] == "backward"
    monkeypatch.setenv("RANK", "1")
    assert bench.run_bwd_reference(args, bench.workload("tiny")) is None
    assert capsys.readouterr().out == ""
