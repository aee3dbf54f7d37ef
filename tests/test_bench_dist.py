"""bench.py's multi-rank path on the CPU: two gloo ranks (no GPU).

bench.py runs one rank per GPU under torchrun. Every rank times its own replica of the sweep, and
the job's time is the slowest rank's (a MAX all-reduce). Only rank 0 prints, and the reference arm
runs on rank 0 alone. These tests run those pieces with two CPU processes over gloo.
"""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_slowest_rank_over_two_gloo_ranks():
    import _dist_worker
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dist_worker.run, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[:4] for r in results] == [(0, 0, 2, 0), (1, 1, 2, 1)]   # rank, RANK, WORLD_SIZE, LOCAL_RANK
    assert all(r[4] == 15.5 for r in results)                        # every rank gets the slowest time


def test_slowest_rank_without_a_group_is_the_identity():
    assert bench.slowest_rank(12.25, None) == 12.25


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class Args:   # never read on rank 1
        steps = warmup = 1
    bench.run_reference(Args(), rank=1, world=2)
    assert capsys.readouterr().out == ""
