"""The bench's N-replica path on CPU (gloo, world size 2): replicas decode
different tokens, the job time is the slowest rank's, the whole-job value counts
every rank's tokens, and the reference arm runs on rank 0 only."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slower replica
        m = bench.max_over_ranks(torch, dist, local_ms, "cpu")
        out[rank] = (m, bench.job_throughput(8, world, m))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    world = 2
    mgr = mp.get_context("spawn").Manager()  # no fork of this (threaded) process
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1]
    m, v = out[0]
    assert m == 15.0
    assert v == pytest.approx(8 * 2 / 0.015)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(torch, dist, 3.5, "cpu") == 3.5
    assert bench.job_throughput(4, 1, 2.0) == pytest.approx(2000.0)


def test_replica_seeds_are_disjoint():
    base = tuple(range(100))
    seen = set()
    for r in range(8):
        s = set(bench.rank_seeds(base, r))
        assert len(s) == len(base) and not (s & seen)
        seen |= s


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
