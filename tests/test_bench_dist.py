"""The multi-process path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The benchmark runs one replica per GPU (the path shards over batch and heads
with no exchange), so the only cross-rank steps are the barrier and the
max-over-ranks timing; the whole-job value is every rank's units over the
slowest rank's time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    ws, r, local = bench.dist_setup()
    assert (ws, r) == (world, rank)
    bench.barrier(ws)
    local_ms = 100.0 * (rank + 1)          # rank 1 is the slow one
    value, ms = bench.whole_job_rate(1000.0, local_ms, ws, "cpu")
    out[rank] = (value, ms)
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_on_the_slowest_rank():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        value, ms = res[rank]
        assert ms == pytest.approx(200.0)
        assert value == pytest.approx(2 * 1000.0 / 0.2)
