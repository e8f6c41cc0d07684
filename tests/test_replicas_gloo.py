"""The multi-GPU path is replicas only: each rank runs the whole operation on
its own batch and the ranks exchange nothing but the final timing.  These
tests run bench.py's cross-rank helpers in two CPU processes over gloo: every
rank must get the slowest rank's time, and the whole-job value must count all
ranks' work over that time."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.rank_env()
        ms = bench.slowest_rank_ms(times[rank], w)
        value = bench.job_tflops(4.5e10, 10, ms, w)
        out_q.put((r, lr, w, ms, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    world, times = 2, [12.5, 20.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    for r, (rank, lrank, w, ms, value) in enumerate(results):
        assert (rank, lrank, w) == (r, r, world)
        assert ms == max(times)  # every rank sees the slowest rank's time
        assert value == pytest.approx(world * 4.5e10 * 10 / (max(times) * 1e-3) / 1e12)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(7.0, 1) == 7.0
    assert bench.job_tflops(1e12, 1, 1000.0, 1) == pytest.approx(1.0)
