"""The host logic of the multi-process benchmark on CPU: gloo ranks (world
size 2) reduce their step times to the slowest rank, the job value counts
every rank's work over that time, and the reference arm runs on rank 0 only.
"""
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.slowest_rank(torch, dist, times[rank], "cpu")
    finally:
        dist.destroy_process_group()


def test_slowest_rank_over_gloo():
    import torch.multiprocessing as mp
    world = 2
    times = [[1.5, 4.0], [2.25, 3.0]]   # rank 1 has the slower step, rank 0 the slower e2e
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == [2.25, 4.0] and out[1] == [2.25, 4.0]


def test_job_value_counts_every_rank():
    # two ranks doing 1e12 FLOP each, slowest step 2 ms -> 1 PF/s for the job
    assert bench.job_pflops(1e12, 2, 2.0) == pytest.approx(1.0)
    assert bench.job_pflops(1e12, 1, 2.0) == pytest.approx(0.5)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    args = bench.parse()
    assert bench.reference_arm(args) == 0
    assert capsys.readouterr().out == ""
