"""The benchmark's multi-rank path (one process per GPU, sequences sharded, no
collective on the data path) on CPU: two gloo ranks, the slowest rank's time
and the sum of the sequences make the whole-job throughput."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    value, ms = bench.aggregate(100.0 * (rank + 1), 32 * 10, world)
    out[rank] = (value, ms)
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    port = _free_port()
    world = 2
    with mp.get_context("spawn").Manager() as m:  # no fork of a process that may hold threads
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        value, ms = res[rank]
        assert ms == pytest.approx(200.0)
        assert value == pytest.approx(2 * 320 / 0.2)
