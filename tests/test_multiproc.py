"""The benchmark's multi-process path on CPU (world size 2, gloo, 127.0.0.1).

The layer shards over tokens with no data-path exchange (replicas), so the only
cross-rank steps are the barrier and the max-over-ranks of the step time; the
reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env()[:2] == (world, rank)
        dist.barrier()
        ms = bench.max_over_ranks(1.5 + rank)  # rank-dependent step times
        results[rank] = (ms, bench.replica_throughput(world, 8192, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput_with_gloo():
    world = 2
    with mp.get_context("spawn").Manager() as m:  # no fork: the process may hold threads
        results = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        got = dict(results)
    # every rank sees the slowest rank's time; the job value counts both replicas' tokens
    assert got[0][0] == got[1][0] == 2.5
    assert got[0][1] == got[1][1] == pytest.approx(2 * 8192 / 2.5e-3)


def test_max_over_ranks_without_a_process_group_is_identity():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.25) == 3.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    # under torchrun the reference arm's other ranks exit 0 without work
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "oracle_step", lambda *a, **k: called.append(1))

    class Args:
        config, steps, warmup, noisy, int8 = "tiny", 1, 1, False, False

    assert bench.run_reference(Args()) == 0
    assert called == []
