"""Multi-rank host logic of bench.py on CPU (gloo, world_size 2).

The routing path has no exchange step between GPUs: N GPUs run N independent
replicas, and the only cross-rank operations are the barrier and the max of
the per-rank step times.  This checks that aggregation with two gloo ranks.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [0.25, 0.4][rank]          # rank 1 is the slow replica
        ms = bench.reduce_max(local_ms, dist)
        dist.barrier()
        out[rank] = (ms, bench.job_throughput(4096, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_max_and_throughput():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    ms, value = out[0]
    assert ms == pytest.approx(0.4)
    assert value == pytest.approx(2 * 4096 / 0.4e-3)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(1.5, None) == 1.5
    assert bench.job_throughput(4096, 1, 0.2) == pytest.approx(4096 / 0.2e-3)
