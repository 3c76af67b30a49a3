"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the per-step time is the
slowest rank's, and the job throughput counts every rank's units once."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]
    got = bench.max_over_ranks(ms, world, torch.device("cpu"))
    thr = bench.job_throughput(1000, world, got)
    out[rank] = (got, thr)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_throughput_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    got, thr = res[0]
    assert got == 5.0                          # the slower rank sets the step time
    assert thr == pytest.approx(2 * 1000 / 5e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(4.0, 1, None) == 4.0
    assert bench.job_throughput(10, 1, 2.0) == pytest.approx(5000.0)
