"""The bf16 parity bars reject the slips a block kernel could plausibly make (CPU only).

Each slip is planted in the oracle (monkeypatch on one of its functions, or one modulation
vector scaled) at klein width over a 128-token sequence.  The planted block's output,
rounded to bf16 as the GPU's is, is compared with the unplanted oracle through the
figures and bars the GPU block tests use (helpers.block_metrics, BF16_BARS and
BF16_ROWCOL_BARS).  Every slip must fail them; the unplanted oracle, rounded the same
way, passes.  The slips, each a kernel-level mistake:
- RoPE applied to q but not k;
- the RoPE table read one token off;
- the softmax taking exp of log2-scaled scores (log2 e folded in, then a natural
  exponential);
- the last 8 keys of a ragged tail masked out;
- two heads' outputs written to each other's columns;
- a gate 5 % (single-stream) or 10 % (dual-stream attention residual) off.
The whole-output cosine alone (0.999) misses all of them (0.9999 and above): max_abs and
the per-row / per-column errors of the update catch them.
"""
import numpy as np
import pytest
import torch

from oracle import dit_oracle as O
from diffusion_transformer_step_gb300 import synth
import helpers as Hx

BARS = {**Hx.BF16_BARS, **Hx.BF16_ROWCOL_BARS}


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).double().numpy()


def _rope_q_only(real):
    calls = {"n": 0}

    def f(x, cos, sin):  # both block forms rotate q first, then k
        calls["n"] += 1
        return real(x, cos, sin) if calls["n"] % 2 == 1 else x
    return f


def _rope_table_one_token_off(real):
    return lambda x, cos, sin: real(x, np.roll(cos, 1, axis=0), np.roll(sin, 1, axis=0))


def _natural_exp_of_log2_scores(real):
    return lambda q, k, v, q_chunk=2048: real(q * np.log2(np.e), k, v, q_chunk)


def _last_keys_masked(real):
    return lambda q, k, v, q_chunk=2048: real(q, k[:, :-8], v[:, :-8], q_chunk)


def _heads_0_1_swapped(real):
    def f(q, k, v, q_chunk=2048):
        o = real(q, k, v, q_chunk).copy()
        o[:, :, [0, 1]] = o[:, :, [1, 0]]
        return o
    return f


SLIPS = [("rope_on_q_only", "apply_rope", _rope_q_only),
         ("rope_table_one_token_off", "apply_rope", _rope_table_one_token_off),
         ("natural_exp_of_log2_scores", "attention", _natural_exp_of_log2_scores),
         ("last_8_keys_masked", "attention", _last_keys_masked),
         ("heads_0_1_swapped", "attention", _heads_0_1_swapped),
         ("gate_off", None, None)]


@pytest.fixture(scope="module")
def klein_128():
    wd = synth.KLEIN
    wl = synth.Workload("klein_128", wd, 1, 64, (8, 8), ())
    g = synth.generator(0)
    img, txt, sgl = synth.stream_weights(wd, g), synth.stream_weights(wd, g), synth.single_weights(wd, g)
    bi = synth.block_inputs(wl, 0)
    dt = np.float32
    cfg = Hx.oracle_config(wd)
    c, s = O.rope_table(O.token_ids(wl.n_txt, *wl.grid))
    x, m = Hx.to_np(bi["x"], dt), O.split_modulation(Hx.to_np(bi["mod"], dt), wd.hidden)
    wi, wt, wsg = Hx.oracle_stream(img, dt), Hx.oracle_stream(txt, dt), Hx.oracle_single(sgl, dt)
    run = {"single": lambda mod: O.single_block(x, wsg, mod, c.astype(dt), s.astype(dt), cfg, dt),
           "dual": lambda mod: O.dual_block(x, wl.n_txt, wi, wt, mod, c.astype(dt), s.astype(dt), cfg, dt)}
    want = {k: f(m) for k, f in run.items()}
    return x, m, run, want


@pytest.mark.parametrize("kind", ["single", "dual"])
def test_unplanted_oracle_passes_the_bars(klein_128, kind):
    x, m, run, want = klein_128
    mm = Hx.block_metrics(_bf16(want[kind]), want[kind], x)
    assert not Hx.block_metrics_fail(mm, BARS), mm


@pytest.mark.parametrize("kind", ["single", "dual"])
@pytest.mark.parametrize("name,attr,variant", SLIPS, ids=[s[0] for s in SLIPS])
def test_bf16_bars_reject_a_planted_slip(monkeypatch, klein_128, kind, name, attr, variant):
    x, m, run, want = klein_128
    mod = m
    if attr is None:  # one gate vector off: the single block's gate, the dual image stream's attention gate
        key, factor = ("single_gate", 1.05) if kind == "single" else ("img_gate_a", 1.1)
        mod = dict(m)
        mod[key] = m[key] * factor
    else:
        monkeypatch.setattr(O, attr, variant(getattr(O, attr)))
    got = _bf16(run[kind](mod))
    mm = Hx.block_metrics(got, want[kind], x)
    bad = Hx.block_metrics_fail(mm, BARS)
    print(kind, name, {k: round(v, 5) for k, v in mm.items()}, bad)
    assert bad, (kind, name, mm)
    assert mm["cos"] >= Hx.BF16_BARS["cos"]  # the whole-output cosine alone would not see it
