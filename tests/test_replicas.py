"""The multi-GPU path of the benchmark is replicas: one process per GPU, no
data-path collective, the slowest rank's time and every rank's units.  These
tests run that host logic as world_size-2 gloo process groups on the CPU, and
check that the reference arm does its work on rank 0 only."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        # rank r took 10 + 5 r ms for 100 + r tokens
        ms, units = bench.over_ranks(10.0 + 5 * rank, 100 + rank, world, device="cpu")
        q.put((rank, ms, units))
    finally:
        dist.destroy_process_group()


def test_over_ranks_max_time_and_summed_units_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    # every rank sees the slowest time (15 ms) and all 201 tokens
    assert got == [(0, 15.0, 201.0), (1, 15.0, 201.0)]
    assert 201.0 / (15.0 / 1e3) == pytest.approx(13400.0)


def test_over_ranks_one_process_is_local():
    assert bench.over_ranks(12.5, 64, 1) == (12.5, 64.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    # a non-zero rank returns before any oracle work (no process group needed)
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.run_reference(bench.parse()) is None
