"""The N>1 bench path on the CPU: two gloo ranks (one process each, as torchrun launches
them) reduce their step times to the slowest rank, report the whole-job rate, and the
reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        # Rank r "measured" 10 + r ms per step and 2 + 3r ms end to end.
        step_ms = bench.max_over_ranks(10.0 + rank, world)
        e2e_ms = bench.max_over_ranks(2.0 + 3.0 * rank, world)
        rate = bench.whole_job_rate(world, 64, step_ms)
        out[rank] = (step_ms, e2e_ms, rate)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in range(world):
        step_ms, e2e_ms, rate = res[rank]
        assert step_ms == 11.0 and e2e_ms == 5.0
        assert rate == pytest.approx(2 * 64 / 11.0e-3)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(1, 64, 0.5) == pytest.approx(128000.0)


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    import bench

    class Args:
        warmup, steps, gpus = 0, 1, 2

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(Args, None)   # a non-zero rank returns before touching the case
    assert capsys.readouterr().out == ""
