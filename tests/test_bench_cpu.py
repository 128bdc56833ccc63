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


def test_hbm_class_bytes_of_the_1024_step():
    """adaLN: 5 dual blocks x (bf16 pass 4NH + fp32-input pass 6NH) + 20 single x 4NH + the
    final pass over the 4096 target rows (4 x 4096 x H); modulation: the 256->H, H->H and
    H->17H weights in bf16.  N = 4608, H = 3072."""
    wl = synth.WORKLOADS["step_1024"]
    b = bench.step_class_bytes(wl.widths, wl.batch, wl.n_txt, wl.n_img, wl.n_ref)
    assert b["adaln"] == 707_788_800 + 1_132_462_080 + 50_331_648
    assert b["modulation_gemv"] == 341_311_488
    b4 = bench.step_class_bytes(wl.widths, 4, wl.n_txt, wl.n_img, wl.n_ref)
    assert b4["adaln"] == 4 * b["adaln"] and b4["modulation_gemv"] == b["modulation_gemv"]


def test_kernel_breakdown_rates_and_shares():
    recs = {"adaln": [0.02] * 62, "gemm_fused_qkv_mlp": [0.43] * 40, "attention": [0.2] * 50}
    flops = {"gemm_fused_qkv_mlp": 7.83e11, "attention": 2.609e11}
    k = bench.kernel_breakdown(recs, flops, {"adaln": 1.8906e9}, 2, 6800.0)
    assert k["adaln"]["launches"] == 62 and k["adaln"]["ms_total"] == pytest.approx(1.24)
    assert k["adaln"]["gbs"] == pytest.approx(1.8906e9 * 2 / 1.24e-3 / 1e9, abs=0.1)
    assert k["adaln"]["frac_of_hbm"] == pytest.approx(k["adaln"]["gbs"] / 6800.0, abs=1e-4)
    assert "tflops" not in k["adaln"] and "gbs" not in k["attention"]
    assert k["gemm_fused_qkv_mlp"]["tflops"] == pytest.approx(7.83e11 / 0.43e-3 / 1e12, abs=0.1)
    assert sum(v["share"] for v in k.values()) == pytest.approx(1.0, abs=1e-3)
    assert bench.kernel_breakdown(recs, flops, {"adaln": 1e9}, 2, None)["adaln"]["frac_of_hbm"] is None


def test_dense_peak_at_clock_and_the_oracle_sample_scaling():
    """The clock-scaled dense peak is SMs x 8192 FLOP per clock x the clock (152 SMs at
    1691 MHz: 2105.6 TFLOP/s), and no clock sample gives none; the CPU sample's scaling to a
    whole step is 5 dual + 20 single block times."""
    class Props:
        multi_processor_count = 152
    p = bench.dense_peak_at_clock(1691.0, Props())
    assert p["tflops"] == pytest.approx(152 * 8192 * 1691e6 / 1e12, abs=0.05) and p["sms"] == 152
    assert bench.dense_peak_at_clock(None, Props()) is None
    wl = synth.WORKLOADS["tiny"]
    calls = []

    def fake_blocks(w, seed=0):
        assert w is wl
        return lambda: calls.append(1) or (2.0, 3.0)

    orig = bench.oracle_blocks
    bench.oracle_blocks = fake_blocks
    try:
        smp = bench.oracle_sample(wl, reps=2)
    finally:
        bench.oracle_blocks = orig
    nd, ns = wl.widths.n_dual, wl.widths.n_single
    assert len(calls) == 2 and smp["dual_block_s"] == 2.0 and smp["single_block_s"] == 3.0
    assert smp["step_s_scaled"] == nd * 2.0 + ns * 3.0 and smp["sample_s"] == 5.0
