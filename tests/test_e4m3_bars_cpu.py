"""The e4m3 parity bars reject a wrong scale (CPU only, no GPU).

A copy of the oracle's quantised linear with one planted mistake -- one output column's
weight scale, or one token row's activation scale, 25 % off, in the last projection of a
klein-width block (the single-stream out-projection over [attn | act], the image stream's
MLP-out of a dual-stream block) -- must fail the bars the GPU parity tests apply to the
e4m3 path, when compared with the unplanted oracle the way the GPU result is (its output
rounded to bf16).  A 25 % error is what a scale taken from another row or column of the
same tensor typically gives.  The unplanted oracle, rounded the same way, passes them.
The column is one whose update is of median size: a column whose update lies below the
bf16 output's resolution cannot show any mistake.
"""
import numpy as np
import pytest
import torch

from oracle import dit_oracle as O
from diffusion_transformer_step_gb300 import synth
import helpers as Hx

BARS = {**Hx.E4M3_BARS, **Hx.E4M3_ROWCOL_BARS}


def _planted_linear(real, target, kind, idx, factor=1.25):
    """A scratch copy of linear_e4m3 that mis-scales one output column (kind "col") or one
    token row (kind "row") when it projects with the weight array `target`."""
    def lin(a, w, dtype=np.float64):
        if w is not target:
            return real(a, w, dtype)
        qa, sa = O.quantize_rows_e4m3_values(a)
        qw, sw = O.quantize_rows_e4m3_values(w)
        sa, sw = sa.copy(), sw.copy()
        if kind == "col":
            sw[idx] *= factor
        else:
            sa.reshape(-1)[idx] *= factor
        return (qa.astype(dtype) @ qw.astype(dtype).T) * sa[..., None].astype(dtype) * sw.astype(dtype)
    return lin


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("kind", ["single", "dual"])
def test_e4m3_bars_reject_a_wrong_scale(monkeypatch, kind):
    wd = synth.KLEIN
    wl = synth.Workload("klein_128", wd, 1, 64, (8, 8), ())
    g = synth.generator(0)
    img, txt, sgl = synth.stream_weights(wd, g), synth.stream_weights(wd, g), synth.single_weights(wd, g)
    bi = synth.block_inputs(wl, 0)
    dt = np.float32
    cfg = Hx.oracle_config(wd)
    c, s = O.rope_table(O.token_ids(wl.n_txt, *wl.grid))
    c, s = c.astype(dt), s.astype(dt)
    x, m = Hx.to_np(bi["x"], dt), O.split_modulation(Hx.to_np(bi["mod"], dt), wd.hidden)
    wi, wt, wsg = Hx.oracle_stream(img, dt), Hx.oracle_stream(txt, dt), Hx.oracle_single(sgl, dt)
    if kind == "single":
        run, target = (lambda: O.single_block(x, wsg, m, c, s, cfg, dt, e4m3="all")), wsg.out
    else:
        run, target = (lambda: O.dual_block(x, wl.n_txt, wi, wt, m, c, s, cfg, dt, e4m3="all")), wi.mlp_out
    want = run()
    ok = Hx.block_metrics(_bf16(want), want, x)
    assert not Hx.block_metrics_fail(ok, BARS), ok
    u = (_bf16(want) - x)[0]
    col_rms = np.sqrt((u * u).mean(axis=0))
    median_col = int(np.argsort(col_rms)[len(col_rms) // 2])
    # token rows of the projection's own input: the single block's out-projection sees all
    # N rows, the image stream's MLP-out its n_img rows
    for plant, idx in (("col", median_col), ("row", 10), ("row", 50)):
        monkeypatch.setattr(O, "linear_e4m3", _planted_linear(O.linear_e4m3, target, plant, idx))
        got = _bf16(run())
        monkeypatch.undo()
        mm = Hx.block_metrics(got, want, x)
        bad = Hx.block_metrics_fail(mm, BARS)
        print(kind, plant, idx, {k: round(v, 5) for k, v in mm.items()}, bad)
        assert bad, (kind, plant, idx, mm)
        assert ("col_err" in bad) if plant == "col" else ("row_err" in bad)


def test_denoise_loop_passes_e4m3_to_every_step():
    """The oracle's loop with the e4m3 option is the loop of e4m3 steps (the option reaches
    every DiT call; the Euler update stays unquantised), and it differs from the unquantised
    loop: the GPU e4m3 loop test compares against this."""
    wl = synth.WORKLOADS["tiny"]
    logical = synth.model_weights(wl.widths, seed=3)
    inp = synth.step_inputs(wl, seed=3)
    ow = Hx.oracle_weights(wl.widths, logical)
    ids = O.token_ids(wl.n_txt, *wl.grid, wl.ref_grids)
    sig = O.sigma_schedule(float(inp["sigma"][0]))
    x0 = Hx.to_np(inp["img_tokens"])
    txt = Hx.to_np(inp["txt_emb"])
    got = O.denoise(ow, x0, None, txt, ids, sig, e4m3="all")
    x = x0.astype(np.float64)
    for k in range(len(sig) - 1):
        v = O.dit_step(ow, x, None, txt, np.full(wl.batch, sig[k]), ids, e4m3="all")
        x = O.euler_update(x, v, sig[k], sig[k + 1])
    np.testing.assert_array_equal(got, x)
    plain = O.denoise(ow, x0, None, txt, ids, sig)
    assert np.abs(got - plain).max() > 0
