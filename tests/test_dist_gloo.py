"""The multi-process side of bench.py on CPU: two gloo ranks go through the
same Dist set-up, barrier and max-over-ranks as the GPU ranks (replicas
only: no data-path collective), and whole-job throughput uses the slowest
rank's time."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import bench
    d = bench.Dist(backend="gloo")
    d.setup(torch)
    d.barrier()
    slowest = d.max(torch, 10.0 + 5.0 * rank)         # rank 1 is slower
    d.barrier()
    out.put((d.rank, d.world, slowest))
    d.done()


def test_two_gloo_ranks_share_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 15.0), (1, 2, 15.0)]
    # Whole-job throughput as bench.py forms it: work of all ranks over the max time.
    work_per_rank, steps, world, max_ms = 56.73e9, 20, 2, 15.0
    assert work_per_rank * steps * world / (max_ms / 1e3) == pytest.approx(56.73e9 * 40 / 0.015)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import torch
    import bench
    d = bench.Dist(backend="gloo")
    d.setup(torch)
    assert d.world == 1 and d.pg is None and d.max(torch, 3.5) == 3.5
