"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each a replica with its
own time, reduce to the slowest rank and report whole-job steps/s."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [30.0, 45.0][rank]              # per-rank ms per step
    m = bench.reduce_max(ms, world, "cpu")
    v = bench.whole_job_steps_per_s(m, world)
    out[rank] = (m, v)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_reduce_to_slowest_rank():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        m, v = out[r]
        assert m == 45.0
        assert abs(v - 2 / 0.045) < 1e-9


def test_single_rank_identity():
    import bench
    assert bench.reduce_max(12.5, 1, "cpu") == 12.5
    assert abs(bench.whole_job_steps_per_s(25.0, 1) - 40.0) < 1e-12
