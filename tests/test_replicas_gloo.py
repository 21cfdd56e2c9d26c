"""The N-GPU path of the benchmark runs N independent replicas (no data-path
collective): only the clocks are joined (max over ranks) and the whole-job
rate counts every replica's tokens.  Checked here with world_size-2 gloo
process groups on the CPU; the reference arm runs on rank 0 alone."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(times[rank], world, device="cpu")
    rate = bench.whole_job_rate(16, 100, ms, world)
    out[rank] = (ms, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_with_two_gloo_ranks():
    world = 2
    times = [120.0, 150.0]          # ms for 100 steps on each replica
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), times, out), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        ms, rate = out[r]
        assert ms == 150.0
        assert rate == pytest.approx(2 * 16 * 100 / 0.150)


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(16, 10, 2.0, 1) == pytest.approx(80_000.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    saved = sys.argv
    sys.argv = ["bench.py", "--impl", "reference"]
    try:
        args = bench.parse()
    finally:
        sys.argv = saved
    bench.run_reference(args, rank=1, world=2)     # returns without work or output
    assert capsys.readouterr().out == ""
