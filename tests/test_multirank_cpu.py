"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each a replica with its
own time, reduce to the slowest rank and report whole-job steps/s; a replica that dies
between steps makes the other's next collective fail instead of hang."""
import os
import socket
import time

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


def _worker_dies(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    bench.init_replica_group("gloo", timeout_s=10.0)
    if rank == 1:
        os._exit(3)                      # this replica dies between steps: nothing in flight
    t0 = time.monotonic()
    try:
        bench.reduce_max(30.0, world, "cpu")
        out[rank] = ("returned", time.monotonic() - t0)
    except Exception as e:               # gloo reports the lost peer or the timeout
        out[rank] = (type(e).__name__, time.monotonic() - t0)


def test_dead_replica_fails_the_next_collective_of_the_others():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker_dies, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert procs[1].exitcode == 3
    assert procs[0].exitcode == 0, "the surviving rank must not hang"
    what, seconds = out[0]
    print(f"surviving rank: {what} after {seconds:.2f} s")
    assert what != "returned", "a collective with a dead peer must not succeed"
    assert seconds < 60.0


def _worker_stalls(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    bench.init_replica_group("gloo", timeout_s=3.0)
    if rank == 1:
        time.sleep(8.0)                  # alive, but never joins the collective
        os._exit(0)
    t0 = time.monotonic()
    try:
        bench.reduce_max(30.0, world, "cpu")
        out[rank] = ("returned", time.monotonic() - t0)
    except Exception as e:
        out[rank] = (type(e).__name__, time.monotonic() - t0)


def test_stalled_replica_times_out_the_next_collective_of_the_others():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker_stalls, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert procs[0].exitcode == 0, "the waiting rank must not hang"
    what, seconds = out[0]
    print(f"waiting rank: {what} after {seconds:.2f} s")
    assert what != "returned"
    assert 2.0 <= seconds < 8.0          # the group's 3 s timeout, not the stalled peer's exit
