"""The oracle's pins are sensitive: plausible slips, planted one at a time in the oracle
(on the CPU, through monkeypatch), each make named pins of test_oracle_pins.py fail.

A mutation replaces one oracle function by a wrong variant of it: a dropped or extra
term, a wrong sign, a swapped operand, slot or stream, another convention (split-half
RoPE, theta 10 000, [sin | cos]).  For each, the pins listed beside it must fail; the
unmutated oracle passes them all (test_oracle_pins.py itself).  Nothing here runs on a
GPU or touches the CUDA path.
"""
import math

import numpy as np
import pytest

from oracle import dit_oracle as O
import test_oracle_pins as P


# ------------------------------------------------------------------ wrong variants
def _ln_unbiased(real):
    # variance divided by H - 1 instead of H
    return lambda x, eps: real(x, eps) * np.sqrt((x.shape[-1] - 1) / x.shape[-1])


def _ln_no_centring(real):
    # the mean left in: an RMS normalisation in place of LayerNorm
    return lambda x, eps: x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)


def _adaln_no_one(real):
    # scale * LN(x) + shift, the "1 +" dropped
    return lambda x, shift, scale, eps: real(x, shift, scale - 1.0, eps)


def _adaln_shift_scale_swapped(real):
    return lambda x, shift, scale, eps: real(x, scale, shift, eps)


def _rms_no_weight(real):
    return lambda x, w, eps: real(x, np.ones_like(w), eps)


def _rms_one_plus_weight(real):
    return lambda x, w, eps: real(x, 1.0 + w, eps)


def _silu_wrong_sign(real):
    # z / (1 + exp(z)) in place of z / (1 + exp(-z))
    return lambda z: -real(-z)


def _swiglu_gate_up_swapped(real):
    return lambda gate, up: real(up, gate)


def _attention_scale_1_over_d(real):
    return lambda q, k, v, q_chunk=2048: real(q / math.sqrt(q.shape[-1]), k, v, q_chunk)


def _attention_unscaled(real):
    return lambda q, k, v, q_chunk=2048: real(q * math.sqrt(q.shape[-1]), k, v, q_chunk)


def _attention_k_v_swapped(real):
    return lambda q, k, v, q_chunk=2048: real(q, v, k, q_chunk)


def _rope_reversed_rotation(real):
    return lambda x, cos, sin: real(x, cos, -sin)


def _rope_split_halves(real):
    # the rotate-half convention: pair j is (x[j], x[j + D/2]) instead of (x[2j], x[2j+1])
    def f(x, cos, sin):
        h = x.shape[-1] // 2
        x0, x1 = x[..., :h], x[..., h:]
        c, s = cos[:, None, :], sin[:, None, :]
        return np.concatenate([x0 * c - x1 * s, x0 * s + x1 * c], axis=-1)
    return f


def _rope_theta_10000(real):
    return lambda ids, axes_dim=(32, 32, 32, 32), theta=2000.0: real(ids, axes_dim, 10000.0)


def _rope_axes_reversed(real):
    # axis a reads id column 3 - a: (l, w, h, t) in place of (t, h, w, l)
    return lambda ids, axes_dim=(32, 32, 32, 32), theta=2000.0: real(np.asarray(ids)[:, ::-1], axes_dim, theta)


def _sinusoid_sin_first(real):
    def f(sigma, dim=256, max_period=10000.0):
        r = real(sigma, dim, max_period)
        return np.concatenate([r[:, dim // 2:], r[:, :dim // 2]], axis=1)
    return f


def _sinusoid_no_1000(real):
    return lambda sigma, dim=256, max_period=10000.0: real(np.asarray(sigma, dtype=np.float64) / 1000.0, dim,
                                                            max_period)


def _modulation_no_last_silu(real):
    # m = W_mod e instead of W_mod SiLU(e)
    def f(sigma, w_t_in, w_t_out, w_mod, cfg, dtype=np.float64):
        emb = O.timestep_sinusoid(sigma, cfg.time_dim, cfg.time_max_period).astype(dtype)
        e = O.silu(emb @ w_t_in.astype(dtype).T) @ w_t_out.astype(dtype).T
        return e @ w_mod.astype(dtype).T
    return f


def _slots(real, edit):
    def f(m, hidden):
        d = dict(real(m, hidden))
        edit(d)
        return d
    return f


def _swap(d, a, b):
    d[a], d[b] = d[b], d[a]


def _mod_shift_scale_order(real):
    def edit(d):
        for s in ("img_", "txt_"):
            for t in ("_a", "_m"):
                _swap(d, f"{s}shift{t}", f"{s}scale{t}")
        _swap(d, "single_shift", "single_scale")
        _swap(d, "final_shift", "final_scale")
    return _slots(real, edit)


def _mod_streams_swapped(real):
    def edit(d):
        for k in ("shift_a", "scale_a", "gate_a", "shift_m", "scale_m", "gate_m"):
            _swap(d, f"img_{k}", f"txt_{k}")
    return _slots(real, edit)


def _mod_one_plus_gate(real):
    def edit(d):
        for k in list(d):
            if "gate" in k:
                d[k] = 1.0 + d[k]
    return _slots(real, edit)


def _mod_attention_mlp_slots_swapped(real):
    def edit(d):
        for s in ("img_", "txt_"):
            for k in ("shift", "scale", "gate"):
                _swap(d, f"{s}{k}_a", f"{s}{k}_m")
    return _slots(real, edit)


def _euler_wrong_sign(real):
    return lambda x, v, sigma_cur, sigma_next: real(x, -v, sigma_cur, sigma_next)


def _qk_rope_before_norm(real):
    # the single-stream block rotating q and k before their RMSNorm
    def f(q, k, qn, kn, cos, sin, cfg):
        q = O.apply_rope(O._heads(q, cfg.heads, cfg.head_dim), cos, sin)
        k = O.apply_rope(O._heads(k, cfg.heads, cfg.head_dim), cos, sin)
        return O.rms_norm(q, qn, cfg.eps), O.rms_norm(k, kn, cfg.eps)
    return f


# (mutation, oracle attribute, wrong variant, pins of test_oracle_pins.py that must fail)
MUTATIONS = [
    ("layer_norm_unbiased", "layer_norm", _ln_unbiased, ["test_layer_norm_moments"]),
    ("layer_norm_no_centring", "layer_norm", _ln_no_centring, ["test_layer_norm_moments"]),
    ("adaln_no_one_plus_scale", "adaln", _adaln_no_one, ["test_adaln_zero_modulation_is_library_layer_norm"]),
    ("adaln_shift_scale_swapped", "adaln", _adaln_shift_scale_swapped, ["test_adaln_shift_and_one_plus_scale"]),
    ("rms_norm_no_weight", "rms_norm", _rms_no_weight, ["test_rms_norm_against_library_and_constant_weight"]),
    ("rms_norm_one_plus_weight", "rms_norm", _rms_one_plus_weight,
     ["test_rms_norm_against_library_and_constant_weight"]),
    ("silu_wrong_sign", "silu", _silu_wrong_sign, ["test_silu_and_swiglu"]),
    ("swiglu_gate_up_swapped", "swiglu", _swiglu_gate_up_swapped,
     ["test_silu_and_swiglu", "test_blocks_mlp_gate_is_the_first_half"]),
    ("attention_scale_1_over_d", "attention", _attention_scale_1_over_d,
     ["test_attention_brute_force_tiny", "test_attention_against_library_sdpa_and_heads_separate"]),
    ("attention_unscaled", "attention", _attention_unscaled, ["test_attention_brute_force_tiny"]),
    ("attention_k_v_swapped", "attention", _attention_k_v_swapped, ["test_attention_brute_force_tiny"]),
    ("rope_reversed_rotation", "apply_rope", _rope_reversed_rotation,
     ["test_rope_matches_complex_rotation_with_pages_constants"]),
    ("rope_split_halves", "apply_rope", _rope_split_halves,
     ["test_rope_axis_ownership_and_adjacent_pairs", "test_rope_preserves_every_pair_norm"]),
    ("rope_theta_10000", "rope_angles", _rope_theta_10000, ["test_rope_frequency_ladder_fixes_theta"]),
    ("rope_axes_reversed", "rope_angles", _rope_axes_reversed, ["test_rope_axis_ownership_and_adjacent_pairs"]),
    ("sinusoid_sin_first", "timestep_sinusoid", _sinusoid_sin_first, ["test_sinusoid_closed_forms"]),
    ("sinusoid_without_1000", "timestep_sinusoid", _sinusoid_no_1000, ["test_sinusoid_closed_forms"]),
    ("modulation_no_last_silu", "modulation", _modulation_no_last_silu,
     ["test_modulation_closed_form_at_sigma_zero"]),
    ("modulation_shift_scale_order", "split_modulation", _mod_shift_scale_order,
     ["test_modulation_slots_and_zero_input_path"]),
    ("modulation_streams_swapped", "split_modulation", _mod_streams_swapped,
     ["test_dual_block_routes_streams_to_their_modulation", "test_modulation_slots_and_zero_input_path"]),
    ("modulation_one_plus_gate", "split_modulation", _mod_one_plus_gate,
     ["test_dual_block_zero_gates_leave_residual_unchanged"]),
    ("modulation_attention_mlp_slots_swapped", "split_modulation", _mod_attention_mlp_slots_swapped,
     ["test_dual_block_mlp_uses_its_own_modulation_slots"]),
    ("euler_wrong_sign", "euler_update", _euler_wrong_sign, ["test_euler_loop_telescopes_and_schedule_ends_at_zero"]),
    ("qk_rope_before_norm", "_qk_norm_rope", _qk_rope_before_norm,
     ["test_dual_and_single_blocks_agree_on_the_attention_path"]),
]


def _fails(pin) -> bool:
    try:
        pin()
    except Exception:  # an assertion, or the wrong variant breaking a shape
        return True
    return False


@pytest.mark.parametrize("name,attr,variant,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_slip_fails_its_pins(monkeypatch, name, attr, variant, pins):
    for p in pins:
        assert not _fails(getattr(P, p)), f"{p} fails on the unmutated oracle"
    monkeypatch.setattr(O, attr, variant(getattr(O, attr)))
    passed = [p for p in pins if not _fails(getattr(P, p))]
    assert not passed, f"mutation {name} passes {passed}"
