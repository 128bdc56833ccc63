"""Host-side checks of the measurement code: the FLOP accounting the roofline and the
TFLOP/s figures use, and the timing hook's argument checks (no GPU)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from diffusion_transformer_step_gb300 import synth  # noqa: E402


@pytest.mark.parametrize("name", ["step_1024", "ref_1920x1088_b4", "tiny"])
def test_class_flops_add_up_to_the_step(name):
    """Per-class FLOPs x launches per step + the embedders and the final projection equal
    the step's FLOPs (multiply-add = 2), and the 1024^2 step is 3.482e13 FLOP."""
    wl = synth.WORKLOADS[name]
    wd = wl.widths
    c = bench.class_flops(wd, wl.batch, wl.n_txt, wl.n_img, wl.n_ref)
    step = bench.step_flops(wd, wl.batch, wl.n_txt, wl.n_img, wl.n_ref)
    blocks = wd.n_single * (c["gemm_fused_qkv_mlp"] + c["gemm_single_out_proj"] + c["attention"]) + wd.n_dual * (
        c["gemm_qkv_rmsnorm_rope"] + c["gemm_dual_out_proj"] + c["gemm_swiglu"] + c["gemm_dual_mlp_out"] +
        c["attention"])
    B, H, C = wl.batch, wd.hidden, wd.in_channels
    embed_final = 2.0 * B * ((wl.n_img + wl.n_ref) * C * H + wl.n_txt * wd.txt_dim * H + wl.n_img * H * C)
    assert step == pytest.approx(blocks + embed_final, rel=1e-12)
    if name == "step_1024":
        assert step == pytest.approx(3.482e13, rel=1e-3)


def test_timing_select_rejects_an_empty_mask():
    from diffusion_transformer_step_gb300 import build_lib
    build_lib.build()
    from diffusion_transformer_step_gb300 import dit
    L = dit.lib()
    assert L.dit_timing_select(0) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_timing_select(0xFFFFFFFF) == dit.DIT_OK
