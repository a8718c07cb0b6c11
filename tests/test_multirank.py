"""The multi-rank host logic of bench.py on CPU ranks (gloo, world size 2,
127.0.0.1): rank discovery from the launcher's environment, the slowest
rank's time shared by every rank, the whole-job value (each rank decodes its
own sequences: weak scaling, no data-path collective), and the reference arm
running on rank 0 alone."""

import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    w, r, lr = bench._dist()
    t = bench._job_seconds(1.0 + 0.5 * rank, "cpu")  # rank 1 is the slow one
    v = bench._job_gbs(40e9, w, t)
    dist.barrier()
    q.put((rank, w, r, lr, t, v))
    dist.destroy_process_group()


def test_two_ranks_share_the_slowest_time_and_sum_the_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r0, w, r, lr, t, v) in enumerate(out):
        assert (r0, w, r, lr) == (rank, 2, rank, rank)
        assert t == 1.5  # the max over ranks, seen by both
        assert v == pytest.approx(2 * 40e9 / 1.5 / 1e9)  # both ranks' bytes in the slowest time
    import bench

    assert bench.aggregate([40e9, 40e9], [1.0, 1.5]) == pytest.approx(out[0][5] * 1e9)


def test_one_rank_keeps_its_own_time():
    sys.path.insert(0, ROOT)
    import bench

    assert bench._job_seconds(0.25, "cpu") == 0.25
    assert bench._job_gbs(10e9, 1, 0.5) == pytest.approx(20.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = type("Args", (), {"workload": "q4_0_mha_1k", "steps": 1, "warmup": 0})()
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""  # no work, no line
