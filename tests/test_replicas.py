"""The multi-GPU path of the benchmark is replicas only: one independent layer per GPU, no
collective on the data path.  Its host logic (barriers around the timed region, the slowest
rank's time, the whole-job rate, rank 0 alone printing) runs here as world_size-2 gloo ranks on
the CPU."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.replica_barrier(world)
        # per-rank step times: the job is as slow as its slowest replica
        ms = bench.replica_max(10.0 + 5.0 * rank, world, "cpu")
        rate = bench.whole_job_rate(4096, world, ms)
        bench.replica_barrier(world)
        q.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_rate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms, rate in got:
        assert ms == 15.0
        assert rate == pytest.approx(4096 * 2 / 15e-3)


def test_single_rank_needs_no_process_group():
    assert bench.replica_max(3.5, 1, "cpu") == 3.5
    bench.replica_barrier(1)
    assert bench.whole_job_rate(4096, 1, 20.0) == pytest.approx(204800.0)


def test_reference_arm_runs_on_rank_0_only():
    """Under torchrun the reference arm (the CPU oracle) runs and prints on rank 0; the other
    ranks return at once without work or output."""
    class A:
        steps, warmup, gpus = 1, 3, 2
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.run_reference(A(), rank=1, world=2)
    assert out.getvalue() == ""
