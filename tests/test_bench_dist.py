"""The benchmark's multi-rank bookkeeping on CPU ranks (gloo, world size 2):
each rank runs an independent replica, the job time is the slowest rank's,
and the throughput counts every rank's work.  Also: the reference arm does
no work on ranks other than 0."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, local_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(local_ms[rank], world)
        out[rank] = (ms, bench.whole_job_tflops(1e12, 5, world, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_with_two_gloo_ranks():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    local_ms = [120.0, 250.0]
    mp.start_processes(_worker, args=(world, port, local_ms, out), nprocs=world, start_method="spawn", join=True)
    for rank in range(world):
        ms, value = out[rank]
        assert ms == 250.0
        # 2 ranks x 5 steps x 1e12 FLOP in 0.25 s = 40 TFLOP/s
        assert value == pytest.approx(40.0)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_tflops(2e12, 4, 1, 1000.0) == pytest.approx(8.0)


def test_reference_arm_does_nothing_off_rank_zero(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    import argparse

    from sequence_blockwise_self_gb300 import inputs

    bench.run_reference(argparse.Namespace(gpus=2, steps=1, warmup=0), inputs.WORKLOADS["tiny"])
    assert capsys.readouterr().out == ""


def test_cpulist_parsing():
    import bench
    assert bench._cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench._cpulist("5") == {5}
    assert bench._cpulist("") == set()


def test_reference_arm_prints_one_contract_line(monkeypatch, capsys):
    """Rank 0 of the reference arm times the oracle and prints one JSON line
    with the keys the benchmark contract names (and no device traffic)."""
    import argparse
    import json

    from sequence_blockwise_self_gb300 import inputs

    monkeypatch.delenv("RANK", raising=False)
    bench.run_reference(argparse.Namespace(gpus=1, steps=1, warmup=0), inputs.WORKLOADS["tiny"])
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("tiny")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
