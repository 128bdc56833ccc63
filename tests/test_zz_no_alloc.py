"""dit_modulation_static, the allocation-free modulation, against dit_modulation.

Callers that cannot allocate device memory where they run the modulation (a plugin whose
host framework owns every device buffer and passes it only its inputs and outputs, or a
serving loop that forbids allocation after start-up) use dit_modulation_static, whose
scratch is a fixed device array inside the library.  It launches the same three kernels
on the same inputs as dit_modulation, only with another scratch address, so its output
must equal the workspace variant's bit for bit, on two calls in a row with different batch
sizes; one call is also checked against the oracle within the modulation tolerance of the
kernel tests (1e-2).  Sizes beyond its fixed maximum must be refused, and a refusal must
leave the next call of the library working.
This file is collected last so that a stop-at-first-failure run has run everything else.
"""
import numpy as np
import pytest
import torch

from diffusion_transformer_step_gb300 import synth
from oracle import dit_oracle as O
import helpers as Hx

pytestmark = pytest.mark.gpu
DEV = "cuda"
ORACLE_TOL = 1e-2


def test_static_modulation_matches_workspace_modulation():
    from diffusion_transformer_step_gb300 import build_lib
    build_lib.build()
    from diffusion_transformer_step_gb300 import dit

    wd = synth.KLEIN
    mw = synth.mod_weights(wd, synth.generator(21))
    dev = {k: v.to(DEV) for k, v in mw.items()}
    w = dit.dit_weights()
    w.cfg = dit.make_config(hidden=wd.hidden, heads=wd.heads, mlp_hidden=wd.mlp_hidden)
    w.mod.t_in, w.mod.t_out, w.mod.mod = dev["t_in"].data_ptr(), dev["t_out"].data_ptr(), dev["mod"].data_ptr()
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)

    def both(sigmas):
        b = len(sigmas)
        sigma = torch.tensor(sigmas, dtype=torch.float32, device=DEV)
        want = torch.empty((b, 17 * wd.hidden), dtype=torch.bfloat16, device=DEV)
        got = torch.full((b, 17 * wd.hidden), float("nan"), dtype=torch.bfloat16, device=DEV)
        dit.dit_modulation(w, sigma, b, want, ws, ws.numel())
        dit.dit_modulation_static(w, sigma, b, got)
        torch.cuda.synchronize()
        return got, want

    for sigmas in ([0.91, 0.37, 0.66], [0.12, 0.99]):     # two calls in a row, different batch
        got, want = both(sigmas)
        assert torch.equal(got, want), (got.float() - want.float()).abs().max().item()

    ref = O.modulation(np.asarray([0.12, 0.99]), Hx.to_np(mw["t_in"]), Hx.to_np(mw["t_out"]), Hx.to_np(mw["mod"]),
                       O.Config(hidden=wd.hidden))
    err = Hx.max_abs(Hx.to_np(got), ref)
    assert err <= ORACLE_TOL, err

    with pytest.raises(dit.DitError) as e:
        dit.dit_modulation_static(w, torch.zeros(9, device=DEV), 9, torch.empty((9, 17 * wd.hidden),
                                                                                dtype=torch.bfloat16, device=DEV))
    assert e.value.status == dit.DIT_ERR_UNSUPPORTED
    # the refusal launched nothing and left no error behind: both variants still run
    got, want = both([0.5])
    assert torch.equal(got, want)
