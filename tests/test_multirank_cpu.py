"""The N > 1 host path of bench.py on CPU: two gloo ranks.

The path does not shard (every rank runs an independent replica), so the
only multi-rank logic is on the host: the job's step time is the slowest
rank's, every rank agrees on it, the whole-job value counts every rank's
work, and rank 0 alone prints (and alone runs the reference arm).
"""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=ws)
    try:
        env = bench.dist_env()
        per_rank_ms = [10.0, 13.5][rank]  # rank 1 is the slow replica
        slowest = bench.max_over_ranks(per_rank_ms, ws, "cpu")
        value = bench.job_value(ws, 2.0e9, slowest)
        q.put((rank, env, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_replica():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort()
    for rank, env, slowest, value in got:
        assert env == (ws, rank, rank)
        assert slowest == pytest.approx(13.5)
        # two replicas' work over the slow replica's time: 2 * 2e9 / 13.5 ms
        assert value == pytest.approx(2 * 2.0e9 / 13.5e-3 / 1e12)


def test_single_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.25, 1, "cpu") == 7.25
    assert bench.job_value(1, 1e12, 1000.0) == pytest.approx(1.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    # a non-zero rank returns before importing or running anything
    assert bench.run_reference(None) is None
