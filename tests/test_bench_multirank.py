"""The benchmark's multi-rank path on CPU: two processes joined by a gloo
process group (as torchrun would launch them, rendezvous on 127.0.0.1) must
agree on the slowest rank's time, report whole-job throughput for weak
scaling, and only rank 0 may run the reference arm.  No GPU is involved."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench._dist()
        ms = bench._max_over_ranks(1.5 + rank, dist, torch.device("cpu"))
        # the reference arm returns at once on every rank but 0
        ran_reference = None
        if r != 0:
            class A:  # noqa: D401 - minimal stand-in for the parsed arguments
                steps, warmup, gpus = 1, 0, world
            bench.run_reference(A())
            ran_reference = False
        q.put((r, w, local, ms, bench._tflops(w, ms), ran_reference))
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_slowest_time_and_whole_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    sys.path.insert(0, ROOT)
    import bench

    for rank, (r, w, local, ms, tflops, ran_reference) in enumerate(res):
        assert (r, w, local) == (rank, 2, rank)
        assert ms == 2.5  # the slower rank's 1.5 + 1
        assert tflops == pytest.approx(2 * bench.STEP_FLOP / 2.5e-3 / 1e12)
    assert res[1][5] is False


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench

    assert bench._max_over_ranks(3.0, None, None) == 3.0
    assert bench._tflops(1, 1.0) == pytest.approx(bench.STEP_FLOP / 1e-3 / 1e12)
