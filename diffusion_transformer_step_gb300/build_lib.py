"""Build the CUDA library in-tree: every .cu under csrc/ compiled in parallel for sm_103a,
linked into diffusion_transformer_step_gb300/libdit.so.  No cmake, no torch extension.

    python -m diffusion_transformer_step_gb300.build_lib [--force]
"""
from __future__ import annotations

import concurrent.futures as cf
import fcntl
import json
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdit.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "dit.h")]


def _stale(target, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _stamp(nvcc, extra_flags) -> dict:
    """What the objects in _build were made with: another host architecture, compiler or
    flag set makes every object stale (object files are not portable between hosts)."""
    return {"machine": platform.machine(), "nvcc": os.path.realpath(nvcc), "flags": ARCH + FLAGS + list(extra_flags)}


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile what is stale and link libdit.so; returns its path.  Processes that build at
    the same time (one per rank) take turns on a lock file, so later ones find the objects
    fresh."""
    os.makedirs(BUILD, exist_ok=True)
    with open(os.path.join(BUILD, "lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            return _build_locked(force, verbose, extra_flags)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _build_locked(force, verbose, extra_flags) -> str:
    nvcc = _nvcc()
    stamp_path = os.path.join(BUILD, "stamp.json")
    stamp = _stamp(nvcc, extra_flags)
    try:
        with open(stamp_path) as f:
            force = force or json.load(f) != stamp
    except (OSError, ValueError):
        force = True
    srcs = _sources()
    headers = [p for p in _deps() if not p.endswith(".cu")]
    jobs = []
    for s in srcs:
        obj = os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")
        if force or _stale(obj, [s] + headers):
            jobs.append((s, obj))

    def compile_one(job):
        src, obj = job
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, cmd, r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for src, cmd, r in ex.map(compile_one, jobs):
                if verbose or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{' '.join(cmd)}\n{r.stderr}")
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]
    if force or jobs or _stale(LIB, objs):
        cmd = [nvcc, *ARCH, "-shared", "-o", LIB + ".tmp", *objs, "-lcudart_static", "-ldl", "-lrt", "-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stderr}")
        os.replace(LIB + ".tmp", LIB)
    with open(stamp_path, "w") as f:
        json.dump(stamp, f)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
