"""Benchmark of one FLUX.2 [klein]-style DiT denoising step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One "step" is one pass of the whole hot path (modulation, embedders, 5 dual-stream and
20 single-stream blocks, final layer) over one batch of synthetic input, through the
C ABI (dit_step_fwd).  The default workload is the 1024x1024 step (512 text + 4096 image
tokens, batch 1).  Prints ONE JSON line on rank 0.

  value      steps/s over the timed region, device-resident inputs (CUDA events on the
             launching stream, synchronised on both sides, max over ranks)
  e2e        the same metric through dit_step_host (replayed from a CUDA graph): pinned host
             inputs copied in and the velocity copied out inside the timed region, the host
             waiting for every step's velocity
  roofline   the dominant kernel class (most device time in an untimed two-step pass that
             records CUDA events around every launch and also gives the per-class `kernels`
             breakdown): its algorithmic FLOPs per launch / its mean launch time, measured
             live in the timed region with CUDA events recorded around that class's launches
             only, on their own stream; `peak` is the measured bf16 burst figure (the timed
             region lasts well under a second), with the sustained figure and the dense
             peak at the run's own median SM clock beside it
  fp8_variant  the same step with every block projection in e4m3 (not the headline)
  cpu_baseline  the CPU oracle (fp32 numpy) timed on a bounded sample (one dual-stream and
             one single-stream block at the same shape); the line gives both measured block
             times and the scaling to the step's 5 + 20 blocks
  --impl reference  times the CPU oracle as the reference arm (rank 0 only): every step is
             the same bounded sample, `ms_per_step` the sample's measured time, `value`
             steps/s scaled from it as above.
  --gpus N   N replicas, one process per GPU, each on its own batch rows (no collective on
             the data path); without WORLD_SIZE in the environment the script starts them
             itself under torch.distributed.run.

Weights are seeded random (no trained checkpoint exists here); the step streams 7.4 GB
of weights per step, far larger than the 129 MB L2, so no L2 flush is needed between
timed steps.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "DiT steps/s at 1024² (512 txt + 4096 img tokens); TFLOP/s vs GB300 bf16 peak"
UNIT = "steps/s"

# Roofline denominators: the measured copy bandwidth and bf16 GEMM throughput in
# MEASURED_PEAKS.json when that file is present, else these fallback figures (one earlier
# GB300 measurement), reported as such.
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Dense bf16 tensor rate of one SM: one M128 N256 K16 tcgen05.mma (2*128*256*16 FLOP) per
# 128 cycles, as measured on sm_103a with one issuing thread per SM (design notes, section 5).
# x the SM count x the SM clock gives the dense peak at a given clock.
BF16_FLOP_PER_CLK_PER_SM = 8192.0

# DRAM traffic per launch of the dominant kernel from one ncu capture (see profiles/);
# None until captured for the current kernel.
NCU_TRAFFIC = {
    # profiles/gemm_fused_qkv_mlp__single_block_1024.md: dram read 205.67 MB + write 153.83 MB
    # for one launch of the same shape as in the step (M 4608, N 27648, K 3072), current kernel
    "gemm_fused_qkv_mlp": 359505920,
}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK), "fallback"


def peak_get(peaks, *names):
    for n in names:
        if n in peaks and isinstance(peaks[n], (int, float)):
            return float(peaks[n])
    return None


# ---------------------------------------------------------------------------------- FLOPs
def class_flops(wd, batch, n_txt, n_img, n_ref):
    """Algorithmic FLOPs (multiply-add = 2) of one launch of each kernel class."""
    H, F, C = wd.hidden, wd.mlp_hidden, wd.in_channels
    N = n_txt + n_img + n_ref
    M = batch * N
    return {
        "gemm_qkv_rmsnorm_rope": 2.0 * M * H * 3 * H,
        "gemm_fused_qkv_mlp": 2.0 * M * H * (3 * H + 2 * F),
        "gemm_dual_out_proj": 2.0 * M * H * H,
        "gemm_swiglu": 2.0 * M * H * 2 * F,
        "gemm_dual_mlp_out": 2.0 * M * F * H,
        "gemm_single_out_proj": 2.0 * M * (H + F) * H,
        "attention": 4.0 * batch * N * N * H,
    }


def step_class_bytes(wd, batch, n_txt, n_img, n_ref):
    """Algorithmic DRAM bytes per step of the HBM-bound kernel classes.
    adaln: every pass reads its input rows once and writes the bf16 output once (the dual
    block's second pass reads the fp32 midpoint residual; the final pass covers the target
    rows only); the per-row modulation vectors are a few KB and not counted.
    modulation_gemv: the timestep-MLP and modulation weights read once (bf16)."""
    H = wd.hidden
    N = n_txt + n_img + n_ref
    row16 = N * H * 2
    adaln = batch * (wd.n_dual * (2 * row16 + (N * H * 4 + row16)) + wd.n_single * 2 * row16
                     + 2 * n_img * H * 2)
    modulation = (H * wd.time_dim + H * H + 17 * H * H) * 2
    return {"adaln": float(adaln), "modulation_gemv": float(modulation)}


def kernel_breakdown(ms_by_class, flops_per_launch, bytes_per_step, n_steps, hbm_peak_gbs):
    """Per kernel class, from its launch times (ms) over n_steps steps: launches, total and
    mean time, share of the device time; TFLOP/s for the contractions (FLOPs per launch /
    mean time) and GB/s with the fraction of the HBM peak for the HBM-bound classes (bytes
    per step x n_steps / total time)."""
    total = sum(sum(v) for v in ms_by_class.values())
    out = {}
    for k, v in ms_by_class.items():
        ms = sum(v)
        e = {"launches": len(v), "ms_total": round(ms, 4), "ms_mean": round(ms / len(v), 5),
             "share": round(ms / total, 4) if total else None}
        if k in flops_per_launch:
            e["tflops"] = round(flops_per_launch[k] / (ms / len(v) / 1e3) / 1e12, 1)
        if k in bytes_per_step and ms > 0:
            e["gbs"] = round(bytes_per_step[k] * n_steps / (ms / 1e3) / 1e9, 1)
            e["frac_of_hbm"] = round(e["gbs"] / hbm_peak_gbs, 4) if hbm_peak_gbs else None
        out[k] = e
    return out


def step_flops(wd, batch, n_txt, n_img, n_ref):
    H, F, C = wd.hidden, wd.mlp_hidden, wd.in_channels
    N = n_txt + n_img + n_ref
    blk = 2.0 * N * H * (4 * H + 3 * F) + 4.0 * N * N * H
    embed = 2.0 * (n_img + n_ref) * C * H + 2.0 * n_txt * wd.txt_dim * H + 2.0 * n_img * H * C
    return batch * ((wd.n_dual + wd.n_single) * blk + embed)


def dense_peak_at_clock(sm_mhz, props):
    """Dense bf16 peak (TFLOP/s) of this GPU at the median SM clock seen during the timed
    region: SMs x BF16_FLOP_PER_CLK_PER_SM x clock.  None without a clock sample."""
    if not sm_mhz:
        return None
    sms = int(props.multi_processor_count)
    return {"tflops": round(sms * BF16_FLOP_PER_CLK_PER_SM * float(sm_mhz) * 1e6 / 1e12, 1), "sms": sms,
            "sm_mhz": float(sm_mhz), "flop_per_clk_per_sm": BF16_FLOP_PER_CLK_PER_SM}


# ---------------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 200 ms) of SM clock and throttle reasons while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for_smi(torch, dev_index):
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return dev_index


# ---------------------------------------------------------------------------------- ranks
PG_TIMEOUT_S = 300.0


def init_replica_group(backend: str, timeout_s: float = PG_TIMEOUT_S) -> None:
    """Process group of the replicas (RANK, WORLD_SIZE and MASTER_* from the environment).
    A replica that dies between steps makes the others' next collective (the barriers
    around the timed region, the max over ranks) end with an error within timeout_s
    instead of waiting without end."""
    import datetime
    import torch.distributed as tdist
    tdist.init_process_group(backend, timeout=datetime.timedelta(seconds=timeout_s))


def reduce_max(x: float, world: int, device) -> float:
    """Max of a per-rank scalar over all ranks (identity at world size 1)."""
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as tdist
        tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def free_port() -> int:
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        return so.getsockname()[1]


def replica_command(n: int, script: str, argv, port: int):
    """The command that runs `script argv` as n ranks of one node under torch.distributed.run,
    rendezvous on 127.0.0.1."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr", "127.0.0.1", "--master-port", str(port), script, *argv]


def relaunch_as_replicas(n: int, script: str, argv) -> int:
    """Start n replicas of this bench (one process per GPU, RANK / LOCAL_RANK / WORLD_SIZE
    set by torch.distributed.run) and return their exit status.  Rank 0 prints the line."""
    return subprocess.call(replica_command(n, script, argv, free_port()))


def whole_job_steps_per_s(ms_per_step_max: float, world: int) -> float:
    """Every rank runs its own replica (its own batch rows): the job completes `world`
    steps in the slowest rank's step time."""
    return world / (ms_per_step_max / 1e3)


def hbm_kernels_alone(torch, dit, W, wl, stream, ws, nbytes, reps=20):
    """Mean time of dit_modulation (the step's batch) and of one bf16 dit_adaln pass over
    the step's B x N rows, each timed alone with CUDA events around `reps` back-to-back
    calls after a warm-up; bytes as in step_class_bytes (weights once; rows read and
    written once)."""
    wd = wl.widths
    H, N, B = wd.hidden, wl.n_tokens, wl.batch
    dev = ws.device
    sigma = torch.full((B,), 0.75, dtype=torch.float32, device=dev)
    mod = torch.empty((B, 17 * H), dtype=torch.bfloat16, device=dev)
    x = torch.randn((B, N, H), device=dev).to(torch.bfloat16)
    y = torch.empty_like(x)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    ms_mod = timed(lambda: dit.dit_modulation(W.w, sigma, B, mod, ws, nbytes, stream))
    ms_ln = timed(lambda: dit.dit_adaln(B, N, H, x, N, 0, N, mod[:, :H], mod[:, H:2 * H], mod[:, :H], mod[:, H:2 * H],
                                        17 * H, 1e-6, y, stream))
    st, where = dit.dit_sync_status(ws, stream)
    if st != dit.DIT_OK:
        raise RuntimeError(f"device wait gave up at site {where:#x}")
    b_mod = (H * wd.time_dim + H * H + 17 * H * H) * 2
    b_ln = 2 * B * N * H * 2
    return {"what": f"each timed alone, {reps} back-to-back calls with CUDA events around them",
            "modulation": {"us_per_call": round(ms_mod * 1e3, 2), "bytes": b_mod,
                           "gbs": round(b_mod / (ms_mod / 1e3) / 1e9, 1)},
            "adaln_bf16": {"us_per_call": round(ms_ln * 1e3, 2), "bytes": b_ln,
                           "gbs": round(b_ln / (ms_ln / 1e3) / 1e9, 1)}}


# ---------------------------------------------------------------------------------- CPU oracle
def oracle_blocks(wl, seed=0):
    """Set up one dual-stream and one single-stream block of the fp32 oracle at wl's shape
    (seeded weights and inputs); returns a function that runs both once and returns the
    seconds each took."""
    import numpy as np
    from diffusion_transformer_step_gb300 import synth
    from oracle import dit_oracle as O

    wd = wl.widths
    g = synth.generator(seed)
    img, txt, sgl = synth.stream_weights(wd, g), synth.stream_weights(wd, g), synth.single_weights(wd, g)
    bi = synth.block_inputs(synth.Workload("b1", wd, 1, wl.n_txt, wl.grid, wl.ref_grids), seed)
    f = lambda t: t.float().numpy()
    cfg = O.Config(hidden=wd.hidden, heads=wd.heads, head_dim=wd.head_dim, mlp_hidden=wd.mlp_hidden)
    sw = lambda d: O.StreamWeights(**{k: f(v) for k, v in d.items()})
    c, s = O.rope_table(O.token_ids(wl.n_txt, *wl.grid, wl.ref_grids))
    c, s = c.astype(np.float32), s.astype(np.float32)
    x, m = f(bi["x"]), O.split_modulation(f(bi["mod"]), wd.hidden)
    wi, wt, ws = sw(img), sw(txt), O.SingleWeights(**{k: f(v) for k, v in sgl.items()})

    def run():
        t0 = time.perf_counter()
        O.dual_block(x, wl.n_txt, wi, wt, m, c, s, cfg, np.float32)
        t1 = time.perf_counter()
        O.single_block(x, ws, m, c, s, cfg, np.float32)
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1

    return run


def oracle_sample(wl, reps=1):
    """The bounded CPU sample both CPU legs time: one dual-stream and one single-stream block
    of the fp32 oracle at wl's shape.  Returns the measured seconds of each and the full
    step's seconds scaled from them (n_dual dual + n_single single blocks; the embedders,
    the modulation and the final layer are under 0.1 % of the step's FLOPs)."""
    run = oracle_blocks(wl)
    td = ts = 0.0
    for _ in range(reps):
        a, b = run()
        td, ts = td + a / reps, ts + b / reps
    wd = wl.widths
    return {"dual_block_s": td, "single_block_s": ts, "sample_s": td + ts,
            "step_s_scaled": wd.n_dual * td + wd.n_single * ts,
            "scaled_to": f"{wd.n_dual} dual + {wd.n_single} single blocks: step_s = {wd.n_dual} t_dual + "
                         f"{wd.n_single} t_single"}


def cpu_cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count()


# ---------------------------------------------------------------------------------- arms
def run_reference(args, wl):
    """The CPU oracle as the reference arm.  Every step is the same bounded sample (one
    dual-stream and one single-stream block of the workload's shape, fp32 numpy); the line's
    ms_per_step is the sample's measured time per step, and value is the workload's steps/s
    scaled from the two measured block times (oracle_sample)."""
    from oracle import dit_oracle as O  # noqa: F401  (the one other place bench runs the oracle)

    wd = wl.widths
    run = oracle_blocks(wl)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    tds, tss = [], []
    for _ in range(args.steps):
        td, ts = run()
        tds.append(td)
        tss.append(ts)
    wall = time.perf_counter() - t0
    td, ts = statistics.mean(tds), statistics.mean(tss)
    step_s = wd.n_dual * td + wd.n_single * ts
    value = wl.batch / step_s
    flops = step_flops(wd, wl.batch, wl.n_txt, wl.n_img, wl.n_ref)
    sample = (f"per step one dual-stream ({td:.2f} s) and one single-stream ({ts:.2f} s) block of the {wl.name} "
              f"shape, fp32 numpy oracle; value scaled to {wd.n_dual} dual + {wd.n_single} single blocks")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(wl), "tflops": flops / step_s / 1e12,
            "sample": {"what": "one dual-stream + one single-stream block per step (ms_per_step is its measured "
                               "time)", "dual_block_s": td, "single_block_s": ts,
                       "step_s_scaled": step_s,
                       "scaled_to": f"{wd.n_dual} t_dual + {wd.n_single} t_single"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(wl):
    return {"workload": wl.name, "batch": wl.batch, "n_txt": wl.n_txt, "n_img": wl.n_img, "n_ref": wl.n_ref,
            "seq_len": wl.n_tokens, "grid": list(wl.grid), "ref_grids": [list(g) for g in wl.ref_grids],
            "l2": "inputs larger than L2 (7.4 GB of bf16 weights streamed per step), no flush",
            "parallelism": "replicas (batch rows per GPU)"}


def run_ours(args, wl, rank, world, local_rank):
    import torch
    import torch.distributed as tdist
    from diffusion_transformer_step_gb300 import build_lib, dit, synth

    build_lib.build()
    dev = f"cuda:{local_rank}"
    torch.cuda.set_device(local_rank)
    wd = wl.widths
    logical = synth.model_weights(wd, seed=rank, device=dev)
    W = dit.DeviceWeights(wd, logical, device=dev)
    del logical
    inp = synth.step_inputs(wl, seed=rank, device=dev)
    shape = dit.make_shape(wl.batch, wl.n_txt, wl.n_img, wl.n_ref)
    ids = dit.dit_token_ids(shape, *wl.grid, wl.ref_grids)
    N = wl.n_tokens
    rope = torch.empty((N, 64, 2), dtype=torch.float32, device=dev)
    dit.dit_rope_table(W.cfg, ids.to(dev), N, rope)
    nbytes = dit.dit_workspace_size(W.cfg, shape)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    vel = torch.empty((wl.batch, wl.n_img, wd.in_channels), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    ref = inp["ref_tokens"]

    def step():
        dit.dit_step_fwd(W.w, shape, inp["img_tokens"], ref, inp["txt_emb"], rope, inp["sigma"], vel, ws, nbytes,
                         stream)

    def barrier():
        if world > 1:
            tdist.barrier()

    for _ in range(args.warmup):
        step()
    st, where = dit.dit_sync_status(ws, stream)
    if st != dit.DIT_OK:
        raise RuntimeError(f"device wait gave up during warm-up at site {where:#x}")

    # ---- per-class breakdown: an untimed pass with an event pair around every launch; it
    #      also names the dominant kernel class, the only one the timed region instruments
    flops_cls = class_flops(wd, wl.batch, wl.n_txt, wl.n_img, wl.n_ref)
    dit.dit_timing_select(0xFFFFFFFF)
    bd_steps = 2
    dit.dit_timing_begin(bd_steps * 200)
    for _ in range(bd_steps):
        step()
    torch.cuda.synchronize()
    bd_records = dit.dit_timing_end(bd_steps * 200)
    bd_by_cls = {}
    for name, t in bd_records:
        bd_by_cls.setdefault(name, []).append(t)
    dom = max((k for k in bd_by_cls if k in flops_cls), key=lambda k: sum(bd_by_cls[k]))
    dom_id = next(i for i in range(32) if dit.dit_kernel_class_name(i) == dom)
    dit.dit_timing_select(1 << dom_id)

    # ---- timed region (device-resident inputs), events around the dominant class's launches
    sampler = ClockSampler(gpu_id_for_smi(torch, local_rank))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = dit.dit_launch_count()
    per_step_launches = None
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    dit.dit_timing_begin(args.steps * 200)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    records = dit.dit_timing_end(args.steps * 200)
    dit.dit_timing_select(0xFFFFFFFF)
    barrier()
    launches = dit.dit_launch_count() - launches0
    ms_total = e0.elapsed_time(e1)
    st, where = dit.dit_sync_status(ws, stream)
    if st != dit.DIT_OK:
        raise RuntimeError(f"device wait gave up in the timed region at site {where:#x}")
    ms_step = reduce_max(ms_total, world, dev) / args.steps
    value = whole_job_steps_per_s(ms_step, world)

    # ---- the HBM-bound kernels timed alone through their entry points (the in-step
    #      breakdown above has an event pair around every one of their short launches):
    #      the whole modulation as one call, and one adaLN pass over the step's rows
    hbm_alone = None
    if rank == 0:
        hbm_alone = hbm_kernels_alone(torch, dit, W, wl, stream, ws, nbytes)

    # ---- host cost of enqueueing one step (direct call, GPU idle before and after)
    host_ms = []
    for _ in range(3):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step()
        host_ms.append((time.perf_counter() - t0) * 1e3)
    torch.cuda.synchronize()

    # ---- the same step replayed from a CUDA graph (one enqueue per step)
    g_dev = dit.dit_step_graph_create(W.w, shape, inp["img_tokens"], ref, inp["txt_emb"], rope, inp["sigma"], vel,
                                      ws, nbytes, host_io=False, stream=stream)
    for _ in range(2):
        dit.dit_graph_launch(g_dev, stream)
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        dit.dit_graph_launch(g_dev, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    graph_ms_step = reduce_max(e0.elapsed_time(e1), world, dev) / args.steps
    dit.dit_graph_destroy(g_dev)

    # ---- the low-precision variant: every block projection in e4m3 (same step otherwise)
    fp8_ms_step = None
    if not args.no_fp8_variant:
        W8 = dit.DeviceWeights(wd, synth.model_weights(wd, seed=rank, device=dev), device=dev, fp8=True)
        step8 = lambda: dit.dit_step_fwd(W8.w, shape, inp["img_tokens"], ref, inp["txt_emb"], rope, inp["sigma"],
                                         vel, ws, nbytes, stream)
        for _ in range(args.warmup):
            step8()
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            step8()
        e1.record(stream)
        torch.cuda.synchronize()
        fp8_ms_step = reduce_max(e0.elapsed_time(e1), world, dev) / args.steps
        del W8, step8
        torch.cuda.empty_cache()

    # ---- e2e through the host-buffer entry point (captured as a graph): every step copies
    # its inputs from pinned host memory, runs, copies the velocity back, and the host waits
    pin = lambda t: t.detach().to("cpu").contiguous().pin_memory() if t is not None else None
    h_img, h_ref, h_txt, h_sig = pin(inp["img_tokens"]), pin(ref), pin(inp["txt_emb"]), pin(inp["sigma"])
    h_vel = torch.empty(tuple(vel.shape), dtype=torch.bfloat16).pin_memory()
    g_host = dit.dit_step_graph_create(W.w, shape, h_img, h_ref, h_txt, rope, h_sig, h_vel, ws, nbytes,
                                       host_io=True, stream=stream)
    for _ in range(2):
        dit.dit_graph_launch(g_host, stream)
        stream.synchronize()
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    k_e2e = max(3, args.steps // 2)
    for _ in range(k_e2e):
        dit.dit_graph_launch(g_host, stream)
        stream.synchronize()  # the caller reads the velocity every step
    e2e_s = reduce_max((time.perf_counter() - t0) / k_e2e, world, dev)
    dit.dit_graph_destroy(g_host)
    h2d = sum(t.numel() * t.element_size() for t in (h_img, h_ref, h_txt, h_sig) if t is not None)
    d2h = h_vel.numel() * h_vel.element_size()

    if rank != 0:
        return

    # ---- roofline of the dominant kernel class (its launches timed inside the timed region)
    peaks, src = load_peaks()
    kernels = kernel_breakdown(bd_by_cls, flops_cls, step_class_bytes(wd, wl.batch, wl.n_txt, wl.n_img, wl.n_ref),
                               bd_steps, peak_get(peaks, "hbm_gbs"))
    dom_ms = [t for name, t in records if name == dom]
    mean_ms = sum(dom_ms) / len(dom_ms)
    achieved = flops_cls[dom] / (mean_ms / 1e3) / 1e12
    peak = peak_get(peaks, "bf16_tflops", "bf16_tflops_sustained")
    peak_sus = peak_get(peaks, "bf16_tflops_sustained")
    clock_peak = dense_peak_at_clock(clocks.get("sm_mhz"), torch.cuda.get_device_properties(local_rank))
    tr = NCU_TRAFFIC.get(dom)
    roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "peak_source": f"bf16 burst, of {src}",
                "traffic": tr, "flops_per_launch": flops_cls[dom], "launch_ms_mean": round(mean_ms, 4),
                "frac_of_sustained": round(achieved / peak_sus, 4) if peak_sus else None,
                "clock_scaled_peak": clock_peak,
                "frac_of_clock_scaled_peak": round(achieved / clock_peak["tflops"], 4) if clock_peak else None}
    if roofline["frac"] > 1.0:
        roofline["note"] = "frac above 1: the denominator (a cuBLAS burst) ran at a lower clock than this kernel"
    flops = step_flops(wd, wl.batch, wl.n_txt, wl.n_img, wl.n_ref)
    tflops = flops / (ms_step / 1e3) / 1e12

    # ---- CPU oracle baseline on a bounded sample (rank 0 of a one-GPU run only)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        smp = oracle_sample(wl)
        cpu = {"value": wl.batch / smp["step_s_scaled"], "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"one dual-stream ({smp['dual_block_s']:.2f} s) and one single-stream "
                         f"({smp['single_block_s']:.2f} s) block of the {wl.name} shape, fp32 numpy oracle, "
                         f"measured once; value scaled to {smp['scaled_to']}",
               "dual_block_s": round(smp["dual_block_s"], 3), "single_block_s": round(smp["single_block_s"], 3),
               "step_s_scaled": round(smp["step_s_scaled"], 2)}

    if hbm_alone is not None and peak_get(peaks, "hbm_gbs"):
        for k in ("modulation", "adaln_bf16"):
            hbm_alone[k]["frac_of_hbm"] = round(hbm_alone[k]["gbs"] / peak_get(peaks, "hbm_gbs"), 4)
    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded random weights and inputs)",
            "config": workload_config(wl),
            "tflops": round(tflops, 1),
            "frac_of_bf16_peak": {"measured_or_fallback": src,
                                  "burst": round(tflops / peak, 4),
                                  "sustained": round(tflops / peak_sus, 4) if peak_sus else None,
                                  "clock_scaled": round(tflops / clock_peak["tflops"], 4) if clock_peak else None},
            "roofline": roofline, "kernels": kernels,
            "kernels_source": f"untimed pass of {bd_steps} steps with an event pair around every launch; the "
                              f"timed region records events around the {dom} launches only",
            "cpu_baseline": cpu,
            "e2e": {"value": round(whole_job_steps_per_s(e2e_s * 1e3, world), 4), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "path": "dit_step_host captured in a CUDA graph, host sync every step"},
            "graph_replay": {"value": round(whole_job_steps_per_s(graph_ms_step, world), 4), "unit": UNIT,
                             "ms_per_step": round(graph_ms_step, 4)},
            "host_enqueue_ms_per_step": round(min(host_ms), 3),
            "fp8_variant": None if fp8_ms_step is None else {
                "what": "every block projection in e4m3 (per-token-row activation and per-output-channel weight "
                        "scales, fp32 accumulation); attention, norms, modulation, embedders and the final "
                        "projection bf16; not the headline",
                "value": round(whole_job_steps_per_s(fp8_ms_step, world), 4), "unit": UNIT,
                "ms_per_step": round(fp8_ms_step, 4)},
            "hbm_kernels_alone": hbm_alone, "gpu_launches": launches, "clocks": clocks}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="step_1024")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8-variant", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    from diffusion_transformer_step_gb300 import synth
    wl = synth.WORKLOADS[args.workload]

    if args.gpus < 1:
        raise SystemExit("--gpus must be >= 1")
    if args.impl == "ours" and args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(relaunch_as_replicas(args.gpus, os.path.abspath(__file__), sys.argv[1:]))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "ours" and world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE {world}: launch one process per GPU")
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, wl)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        init_replica_group("nccl")
    try:
        run_ours(args, wl, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as tdist
            tdist.destroy_process_group()


if __name__ == "__main__":
    main()
