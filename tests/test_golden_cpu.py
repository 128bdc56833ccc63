"""CPU checks of the stored step golden: its inputs are the ones the seeded generators draw
here, and the file is complete (every sampled token of every checked row, 128 channels)."""
import os

import numpy as np
import torch

from diffusion_transformer_step_gb300 import synth
import helpers as Hx

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "step_ref_1920x1088_rows0_3.txt")


def test_ref_step_golden_is_complete():
    kv, vel = Hx.read_step_golden(GOLDEN)
    wl = synth.WORKLOADS["ref_1920x1088_b4"]
    rows = [int(r) for r in kv["rows"].split()]
    toks = [int(t) for t in kv["tokens"].split()]
    assert rows == [0, 3] and toks[0] == 0 and toks[-1] == wl.n_img - 1 and len(set(toks)) == len(toks)
    assert len([float(s) for s in kv["sigma"].split()]) == wl.batch
    assert set(vel) == {(b, t) for b in rows for t in toks}
    for v in vel.values():
        assert v.shape == (wl.widths.in_channels,) and np.isfinite(v).all()
    for b in rows:
        assert float(kv[f"row{b}.rms"]) > 0


def test_ref_step_golden_inputs_match_the_generators():
    """The activations (target, reference and text tokens) drawn here from the golden's seed
    have the fingerprints stored beside the expected velocity; the GPU test checks the weights'."""
    kv, _ = Hx.read_step_golden(GOLDEN)
    wl = synth.WORKLOADS["ref_1920x1088_b4"]
    inp = synth.step_inputs(wl, seed=int(kv["seed"]), draw_dtype=torch.float64)
    Hx.check_fingerprints(Hx.input_fingerprints(None, inp), kv)
    assert inp["img_tokens"].dtype == torch.bfloat16
