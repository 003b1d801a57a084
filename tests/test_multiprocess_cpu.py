"""The N > 1 path of the benchmark on CPU: two gloo ranks, each timing its own
independent sequence (weak scaling). The job's step time is the slowest rank's
and the whole-job value counts every rank's tokens; no data-path collective is
involved (heads and sequences are independent)."""
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


def _worker(rank, world, port, local_ms, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms, value = bench.aggregate(local_ms[rank], 262144, world)
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_weak_scaling_aggregate_two_ranks(world):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    local_ms = [10.0, 12.5]
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, local_ms, out))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    for r in range(world):
        ms, value = out[r]
        assert ms == 12.5  # slowest rank
        assert abs(value - 2 * 262144 / 0.0125) < 1e-6 * value



def test_aggregate_single_process():
    import bench

    ms, value = bench.aggregate(5.0, 1000, 1)
    assert ms == 5.0 and value == pytest.approx(200000.0)
