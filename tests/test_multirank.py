"""The multi-GPU path is replicas only: every rank runs the same seeded
workload on its own GPU with no collective on the data path; the job's time is
the slowest rank's and its throughput the rows of all ranks over that time.
These tests run that host logic as world-size-2 gloo process groups on the CPU
(bench.py's max_over_ranks / job_rows_per_s and the reference arm's rank rule)."""
import hashlib
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench as b
    import workloads as W

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # each replica's step time differs; the job takes the slowest
        ms = [3.0, 5.0][rank]
        ms_max = b.max_over_ranks(ms, dist, torch.device("cpu"))
        # every replica builds the same seeded workload (weak scaling: fixed work per rank)
        wl = W.SMALL["tiny_decode"]()
        h = hashlib.sha256(wl.q.tobytes() + wl.block_tables.tobytes() + wl.hist_k.tobytes()).hexdigest()
        hashes = [None] * world
        dist.all_gather_object(hashes, h)
        results[rank] = (ms_max, b.job_rows_per_s(wl.n_rows, world, ms_max), wl.n_rows, hashes)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_world_2():
    world, port = 2, free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    assert sorted(res) == [0, 1]
    for rank in range(world):
        ms_max, value, rows, hashes = res[rank]
        assert ms_max == 5.0  # the slower replica's time, on both ranks
        assert value == pytest.approx(rows * world / 5e-3)
        assert len(set(hashes)) == 1  # identical seeded inputs on every rank


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(7.25) == 7.25
    assert bench.job_rows_per_s(512, 1, 0.5) == pytest.approx(1.024e6)


def test_reference_arm_runs_on_rank_0_only(monkeypatch, capsys):
    """Under torchrun the other ranks of the reference arm exit without work."""
    called = []
    monkeypatch.setattr(bench, "make_workload", lambda *a, **k: called.append(a) or (_ for _ in ()).throw(
        AssertionError("a rank other than 0 built the workload")))
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"workload": "tiny_decode", "seqs": 0, "warmup": 1, "steps": 1, "gpus": 2})()
    assert bench.run_reference(args) is None
    assert called == [] and capsys.readouterr().out == ""
