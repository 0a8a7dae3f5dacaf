"""The multi-rank host logic of bench.py on CPU: two gloo ranks.

With N GPUs bench.py runs N independent replicas (no collective on the data
path); the only cross-rank steps are the barriers around the timed region and
the reduction of its results: the whole-job rate is the units all ranks
processed divided by the slowest rank's time.  Those reductions are checked
here over gloo, world size 2, on the host.
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: 100 (r + 1) units in 1.5 + r seconds
        units = 100.0 * (rank + 1)
        seconds = 1.5 + rank
        rate, total_s, total_u = bench.job_rate(torch, dist, units, seconds)
        dist.barrier()
        mx = bench.max_over_ranks(torch, dist, float(rank) - 7.0)
        sm = bench.sum_over_ranks(torch, dist, 0.25)
        results[rank] = (rate, total_s, total_u, mx, sm)
    finally:
        dist.destroy_process_group()


def test_job_rate_over_two_gloo_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), results), nprocs=world, join=True,
                       start_method="spawn")
    want_s = 2.5                # the slower rank
    want_u = 100.0 + 200.0      # both ranks' units
    for rank in range(world):
        rate, total_s, total_u, mx, sm = results[rank]
        assert total_s == want_s
        assert total_u == want_u
        assert rate == want_u / want_s
        assert mx == -6.0
        assert sm == 0.5


def test_single_process_reductions_are_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(torch, None, 3.25) == 3.25
    assert bench.sum_over_ranks(torch, None, 3.25) == 3.25
    assert bench.job_rate(torch, None, 10.0, 4.0) == (2.5, 4.0, 10.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup, variant, gpus = 1, 3, "d64", 2

    bench.run_reference(Args(), rank=1, world=2)  # returns at once, prints nothing
    assert capsys.readouterr().out == ""
