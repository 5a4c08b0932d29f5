"""The benchmark's multi-rank path on CPU: two gloo ranks (one process each, as
torchrun launches them) agree on the slowest rank's times, the whole-job value
counts every rank's rows, and the reference arm does its work on rank 0 only."""

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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports step time 1 + r ms and scorer time 10 * (1 + r) ms
        ms, score_ms = bench.max_over_ranks([1.0 + rank, 10.0 * (1 + rank)])
        value = bench.job_rows_per_s(world, 8, ms)
        out[rank] = (ms, score_ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_all_rows():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, score_ms, value = res[rank]
        assert ms == 2.0 and score_ms == 20.0          # the maximum, on every rank
        assert value == pytest.approx(world * 8 / 2e-3)  # 8 rows per rank, slowest rank's time


def test_single_process_aggregation_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.5, 7.0]) == [3.5, 7.0]
    assert bench.job_rows_per_s(1, 8, 0.5) == pytest.approx(16000.0)


def test_reference_arm_does_nothing_off_rank_zero(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    bench.run_reference(bench.parse())
    assert capsys.readouterr().out == ""
