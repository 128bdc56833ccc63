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


def test_bench_gpus_n_starts_n_replicas_itself(monkeypatch):
    """`python bench.py --gpus 2` outside any launcher re-runs itself as 2 ranks under
    torch.distributed.run (rendezvous on 127.0.0.1), passing its own arguments on."""
    import sys
    import bench
    seen = {}

    def fake(n, script, argv):
        seen.update(n=n, script=script, argv=list(argv))
        return 0

    monkeypatch.setattr(bench, "relaunch_as_replicas", fake)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "2", "--steps", "3", "--warmup", "3"])
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert e.value.code == 0
    assert seen["n"] == 2 and seen["script"].endswith("bench.py")
    assert seen["argv"] == ["--gpus", "2", "--steps", "3", "--warmup", "3"]
    cmd = bench.replica_command(2, "/x/bench.py", ["--gpus", "2"], 29500)
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"] and "--nproc-per-node=2" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1" and cmd[-3:] == ["/x/bench.py", "--gpus", "2"]
    # under a launcher, WORLD_SIZE must agree with --gpus
    monkeypatch.setenv("WORLD_SIZE", "4")
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert "WORLD_SIZE 4" in str(e.value.code)


STANDIN = r'''
import json, os, sys, time
sys.path.insert(0, os.environ["BENCH_ROOT"])
import bench
if "WORLD_SIZE" not in os.environ:
    sys.exit(bench.relaunch_as_replicas(2, os.path.abspath(__file__), []))
bench.init_replica_group("gloo", timeout_s=60.0)
import torch.distributed as dist
rank, world = dist.get_rank(), dist.get_world_size()
dist.barrier()
t0 = time.perf_counter()
for _ in range(3):
    time.sleep(0.02 * (rank + 1))          # the stand-in step: rank 1 is the slow replica
ms = (time.perf_counter() - t0) / 3 * 1e3
m = bench.reduce_max(ms, world, "cpu")
if rank == 0:
    print(json.dumps({"n_gpus": world, "ms_per_step": m, "value": bench.whole_job_steps_per_s(m, world),
                      "rank0_ms": ms}), flush=True)
dist.barrier()
dist.destroy_process_group()
'''


def test_replica_launcher_brings_up_two_gloo_ranks(tmp_path):
    """The launcher bench.py uses, run for real with a CPU stand-in step: two ranks come
    up, join one gloo group, and rank 0 alone prints n_gpus 2 and the whole-job rate of
    the slowest rank."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = tmp_path / "standin.py"
    script.write_text(STANDIN)
    env = dict(os.environ, BENCH_ROOT=root, OMP_NUM_THREADS="1")
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, str(script)], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = lines[0]
    assert d["n_gpus"] == 2
    assert d["ms_per_step"] >= 40.0 and d["ms_per_step"] > d["rank0_ms"]      # the slower rank's time
    assert abs(d["value"] - 2 / (d["ms_per_step"] / 1e3)) < 1e-9
