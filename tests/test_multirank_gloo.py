"""Host logic of the multi-rank benchmark on CPU: two ranks over gloo.

One process per GPU runs its own replica of the workload with no data-path
exchange; the only collective is the max of the ranks' timed-region lengths.
These tests run that host logic with a world size of 2 on CPU ranks.
"""
import contextlib
import io
import multiprocessing as mp
import os
import socket
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, seconds, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        sec = bench.slowest_rank_seconds(seconds[rank], world, "cpu")
        q.put((rank, sec, bench.job_gbs(7_110_656 * 2, 10, world, sec)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_rank_and_the_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    seconds = [0.25, 0.5]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, seconds, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    # both ranks see the slowest rank's time, and the value counts both ranks' bytes
    for rank, sec, gbs in got:
        assert sec == 0.5
        assert gbs == pytest.approx(7_110_656 * 2 * 10 * 2 / 0.5 / 1e9)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_seconds(0.125, 1, "cpu") == 0.125
    assert bench.job_gbs(1e9, 4, 1, 2.0) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench
    args = types.SimpleNamespace(steps=1, warmup=0, gpus=2)
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert bench.run_reference(args, rank=1, world=2) is None
    assert out.getvalue() == ""
