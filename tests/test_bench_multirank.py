"""The multi-rank host logic of bench.py on CPU: two gloo ranks reduce their step times to the
slowest rank's, and the whole-job throughput counts every rank's own batch (weak scaling)."""
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
    ms = bench.reduce_max_ms(10.0 + 5.0 * rank, world, "cpu")
    out[rank] = (ms, bench.job_throughput(16384, world, ms))
    dist.destroy_process_group()


def test_two_rank_reduction():
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
    assert out[0][0] == out[1][0] == 15.0
    assert out[0][1] == pytest.approx(2 * 16384 / 0.015)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max_ms(3.5, 1, "cpu") == 3.5
