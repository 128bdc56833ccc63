"""dit_modulation_static, the allocation-free modulation, against dit_modulation.

Callers that cannot allocate device memory where they run the modulation (a plugin whose
host framework owns every device buffer and passes it only its inputs and outputs, or a
serving loop that forbids allocation after start-up) use dit_modulation_static, whose
scratch is a fixed device array inside the library.  Its output must equal the workspace
variant's within the modulation tolerance of the kernel tests (1e-2), on two calls in a
row with different sizes, and sizes beyond its fixed maximum must be refused.
This file is collected last so that a stop-at-first-failure run has run everything else.
"""
import pytest
import torch

from diffusion_transformer_step_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 1e-2


def test_static_modulation_matches_workspace_modulation():
    from diffusion_transformer_step_gb300 import build_lib
    build_lib.build()
    from diffusion_transformer_step_gb300 import dit

    wd = synth.KLEIN
    mw = {k: v.to(DEV) for k, v in synth.mod_weights(wd, synth.generator(21)).items()}
    w = dit.dit_weights()
    w.cfg = dit.make_config(hidden=wd.hidden, heads=wd.heads, mlp_hidden=wd.mlp_hidden)
    w.mod.t_in, w.mod.t_out, w.mod.mod = mw["t_in"].data_ptr(), mw["t_out"].data_ptr(), mw["mod"].data_ptr()
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)

    for sigmas in ([0.91, 0.37, 0.66], [0.12, 0.99]):     # two calls in a row, different batch
        b = len(sigmas)
        sigma = torch.tensor(sigmas, dtype=torch.float32, device=DEV)
        want = torch.empty((b, 17 * wd.hidden), dtype=torch.bfloat16, device=DEV)
        got = torch.full((b, 17 * wd.hidden), float("nan"), dtype=torch.bfloat16, device=DEV)
        dit.dit_modulation(w, sigma, b, want, ws, ws.numel())
        dit.dit_modulation_static(w, sigma, b, got)
        torch.cuda.synchronize()
        err = (got.float() - want.float()).abs().max().item()
        assert err <= TOL, err

    with pytest.raises(dit.DitError) as e:
        dit.dit_modulation_static(w, torch.zeros(9, device=DEV), 9, torch.empty((9, 17 * wd.hidden),
                                                                                dtype=torch.bfloat16, device=DEV))
    assert e.value.status == dit.DIT_ERR_UNSUPPORTED
