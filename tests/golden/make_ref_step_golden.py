"""Write the oracle's expected velocity for the reference-guided batch-4 step.

Workload: a 1920x1088 target (120 wide x 68 high patch grid, 8160 tokens) with one
1024x1024 reference (64x64 grid, t = 10), 512 text rows, N = 12768, klein widths, batch 4
("FLUX.2 [klein] 4B/9B + Z-Image-Turbo on a shared DiT scaffold": reference-guided
editing; rows of a batch are independent).  The fp32 oracle runs the whole 25-block step
for batch rows 0 and 3 only; the GPU test checks the other rows through batch invariance.

What is stored (all from `oracle/`, nothing from the CUDA path):
  * the seed, the per-row sigma and the sampled target tokens;
  * per input tensor group, the float64 sum and sum of squares of the bf16 values that
    the seeded CPU generators produce, so that the test can tell a changed input stream
    from a changed result.  The inputs are drawn in float64 before the bf16 rounding, which
    makes them the same on x86 and Arm hosts (the float32 sampler differs in the last place);
  * per checked row, the mean and rms of the whole velocity [8160, 128];
  * per checked row, the velocity of the sampled tokens (128 channels each).

Run from the repository root (about 30 minutes of CPU on 8 cores, 20 GB of host memory):
    python tests/golden/make_ref_step_golden.py
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

from oracle import dit_oracle as O                      # noqa: E402
from diffusion_transformer_step_gb300 import synth      # noqa: E402
import helpers as Hx                                    # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "step_ref_1920x1088_rows0_3.txt")
SEED = 5
SIGMA = (0.9, 0.7, 0.55, 0.95)
ROWS = (0, 3)
N_SAMPLED_TOKENS = 32


def sampled_tokens(n_img: int) -> np.ndarray:
    return np.unique(np.linspace(0, n_img - 1, N_SAMPLED_TOKENS).round().astype(np.int64))


def main():
    wl = synth.WORKLOADS["ref_1920x1088_b4"]
    t0 = time.time()
    logical = synth.model_weights(wl.widths, seed=SEED, draw_dtype=torch.float64)
    inp = synth.step_inputs(wl, seed=SEED, draw_dtype=torch.float64)
    inp["sigma"] = torch.tensor(SIGMA, dtype=torch.float32)
    fp = Hx.input_fingerprints(logical, inp)
    print(f"inputs {time.time() - t0:.1f} s", flush=True)

    dt = np.float32
    ow = Hx.oracle_weights(wl.widths, logical, dt)
    del logical
    ids = O.token_ids(wl.n_txt, *wl.grid, wl.ref_grids)
    toks = sampled_tokens(wl.n_img)
    lines = [
        "# Expected velocity of the reference-guided batch-4 step (1920x1088 target, one 1024x1024",
        "# reference, 512 text rows, N = 12768, klein widths), batch rows 0 and 3, from the fp32 oracle.",
        "# Written by tests/golden/make_ref_step_golden.py (calls the seeded generators and oracle/ only).",
        "# Inputs: synth.model_weights / step_inputs with draw_dtype float64.",
        f"seed = {SEED}",
        "sigma = " + " ".join(repr(float(s)) for s in SIGMA),
        "rows = " + " ".join(str(r) for r in ROWS),
        "tokens = " + " ".join(str(int(t)) for t in toks),
    ]
    for k, (s, q) in fp.items():
        lines.append(f"fingerprint.{k} = {s!r} {q!r}")
    for b in ROWS:
        t1 = time.time()
        ref = Hx.to_np(inp["ref_tokens"][b:b + 1], dt)
        v = O.dit_step(ow, Hx.to_np(inp["img_tokens"][b:b + 1], dt), ref, Hx.to_np(inp["txt_emb"][b:b + 1], dt),
                       Hx.to_np(inp["sigma"][b:b + 1]), ids, dt)[0].astype(np.float64)
        print(f"row {b}: oracle step {time.time() - t1:.1f} s", flush=True)
        lines.append(f"row{b}.mean = {float(v.mean())!r}")
        lines.append(f"row{b}.rms = {float(np.sqrt((v * v).mean()))!r}")
        for t in toks:
            lines.append(f"v {b} {int(t)} " + " ".join(f"{x:.7g}" for x in v[t]))
    with open(OUT, "w") as f:
        f.write("\n".join(lines) + "\n")
    print(f"wrote {OUT} ({time.time() - t0:.1f} s)")


if __name__ == "__main__":
    main()
