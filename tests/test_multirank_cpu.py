"""The N > 1 host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

Heads are independent, so N GPUs run N replicas with no exchange on the data path;
what the ranks share is the timing: every rank must see the slowest rank's time,
and the reported value counts the work of all ranks over that time.  The reference
arm runs on rank 0 only; the other ranks return without work.
"""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
    val = bench.whole_job_tflops(1e12, 4, world, ms)
    r, w, _ = bench.dist_env()
    q.put((rank, ms, val, r, w))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, val, r, w in out:
        assert ms == 15.0                       # both ranks see the slower rank's 15 ms
        assert abs(val - 1e12 * 4 * 2 / 0.015 / 1e12) < 1e-9
        assert (r, w) == (rank, world)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.5, "cpu") == 7.5
    assert bench.whole_job_tflops(2e12, 10, 1, 20.0) == pytest.approx(1000.0)


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 3, 3

    assert bench.run_reference(A()) is None
