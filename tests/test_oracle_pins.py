"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a wrong
sign, index or axis, a transposed operand, a swapped stream) fails it.  None of them
re-types the oracle's own formula: they use golden values from the pages, closed forms,
invariants, library routines (torch, scipy) for special cases, and brute force.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import dit_oracle as O
from diffusion_transformer_step_gb300 import synth
import helpers as Hx

GOLD = os.path.join(os.path.dirname(__file__), "golden")
STRUCT = Hx.read_kv(os.path.join(GOLD, "klein_structure.txt"))
THETA = float(STRUCT["rope_theta"])
AXIS = int(STRUCT["rope_dims_per_axis"])
AXES = (AXIS,) * int(STRUCT["rope_axes"])
RNG = np.random.default_rng(1234)


# ------------------------------------------------------------------ token ids / RoPE
def test_token_ids_golden_layout():
    want = Hx.read_rows(os.path.join(GOLD, "token_ids_small.txt"))
    got = O.token_ids(3, 2, 3, ref_grids=[(1, 2), (2, 1)])
    np.testing.assert_array_equal(got, want)


def test_token_ids_reference_t_offsets_and_counts():
    n_txt = int(STRUCT["text_rows"])
    first, step = int(STRUCT["ref_t_first"]), int(STRUCT["ref_t_step"])
    ids = O.token_ids(n_txt, 64, 64, ref_grids=[(4, 5), (3, 3), (2, 7)])
    assert ids.shape == (n_txt + 4096 + 20 + 9 + 14, 4)
    ref = ids[n_txt + 4096:]
    assert sorted(set(ref[:, 0].tolist())) == [first, first + step, first + 2 * step]
    assert int(STRUCT["max_references"]) == 3
    # text rows: only the sequence axis moves; image rows: l == 0 and t == 0
    assert (ids[:n_txt, :3] == 0).all() and (ids[:n_txt, 3] == np.arange(n_txt)).all()
    assert (ids[n_txt:n_txt + 4096, [0, 3]] == 0).all()


def _rot(x, ids):
    c, s = O.rope_table(np.asarray(ids, np.float64), AXES, THETA)
    return O.apply_rope(x[None, :, None, :], c, s)[0, :, 0, :]


def test_rope_position_zero_is_identity():
    x = RNG.standard_normal((5, 128))
    np.testing.assert_array_equal(_rot(x, np.zeros((5, 4))), x)


def test_rope_preserves_every_pair_norm():
    x = RNG.standard_normal((7, 128))
    ids = RNG.integers(0, 5000, size=(7, 4))
    y = _rot(x, ids)
    n_in = np.hypot(x[:, 0::2], x[:, 1::2])
    n_out = np.hypot(y[:, 0::2], y[:, 1::2])
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12, atol=1e-12)


def test_rope_matches_complex_rotation_with_pages_constants():
    # Independent route: each adjacent pair is a complex number turned by e^{i*angle},
    # angle = pos_axis * theta^(-2j/32) with the golden theta and axis width.
    x = RNG.standard_normal((6, 128))
    ids = RNG.integers(0, 300, size=(6, 4)).astype(np.float64)
    z = x[:, 0::2] + 1j * x[:, 1::2]
    pos = np.repeat(ids, AXIS // 2, axis=1)                      # pair -> owning axis
    jj = np.tile(np.arange(AXIS // 2), 4)
    zr = z * np.exp(1j * pos * np.power(THETA, -2.0 * jj / AXIS))
    want = np.empty_like(x)
    want[:, 0::2], want[:, 1::2] = zr.real, zr.imag
    np.testing.assert_allclose(_rot(x, ids), want, rtol=1e-10, atol=1e-10)


def test_rope_relative_property():
    q = RNG.standard_normal(128)
    k = RNG.standard_normal(128)
    p = np.array([3, 7, 11, 2], dtype=np.float64)
    pp = np.array([1, 2, 5, 9], dtype=np.float64)
    lhs = _rot(q[None], p[None])[0] @ _rot(k[None], pp[None])[0]
    rhs = _rot(q[None], (p - pp)[None])[0] @ k
    assert abs(lhs - rhs) < 1e-10


def test_rope_axis_ownership_and_adjacent_pairs():
    # A position on axis a only moves dims [32a, 32a+32); dim 2j's partner is 2j+1.
    for a in range(4):
        ids = np.zeros((1, 4)); ids[0, a] = 3.0
        for d in range(0, 128, 2):
            e = np.zeros((1, 128)); e[0, d] = 1.0
            y = _rot(e, ids)[0]
            nz = set(np.flatnonzero(np.abs(y) > 1e-14).tolist())
            if a * AXIS <= d < (a + 1) * AXIS:
                assert nz <= {d, d + 1} and (d + 1 in nz or abs(math.sin(3.0 * THETA ** (-(d - a * AXIS) / AXIS))) < 1e-14)
            else:
                assert nz == {d}


def test_rope_frequency_ladder_fixes_theta():
    # Pair j of an axis at position p turns exactly as pair 0 at position p*theta^(-2j/32):
    # pins theta and the exponent without re-typing the table.
    p = 1000.0
    for j in (1, 5, 8, 15):
        e = np.zeros((1, 128)); e[0, AXIS + 2 * j] = 1.0
        y = _rot(e, np.array([[0, p, 0, 0]]))[0][AXIS + 2 * j: AXIS + 2 * j + 2]
        p_eq = p * THETA ** (-2.0 * j / AXIS)
        z = _rot(np.eye(1, 128), np.array([[p_eq, 0, 0, 0]]))[0][:2]
        np.testing.assert_allclose(y, z, atol=1e-9)
    # and theta is the pages' 2000: pair 8 of axis h at position 2000 turns by sqrt(2000)
    e = np.zeros((1, 128)); e[0, AXIS + 16] = 1.0
    y = _rot(e, np.array([[0, 2000.0, 0, 0]]))[0][AXIS + 16: AXIS + 18]
    np.testing.assert_allclose(y, [math.cos(math.sqrt(2000.0)), math.sin(math.sqrt(2000.0))], atol=1e-9)


# ------------------------------------------------------------------ norms / activations
def test_layer_norm_moments():
    x = RNG.standard_normal((4, 3072)) * 3 + 1.5
    y = O.layer_norm(x, 1e-6)
    np.testing.assert_allclose(y.mean(-1), 0, atol=1e-12)
    var = x.var(-1)
    np.testing.assert_allclose(y.var(-1), var / (var + 1e-6), rtol=1e-12)


def test_adaln_zero_modulation_is_library_layer_norm():
    x = RNG.standard_normal((3, 257))
    z = np.zeros((1, 257))
    want = torch.nn.functional.layer_norm(torch.from_numpy(x), (257,), eps=1e-6).numpy()
    np.testing.assert_allclose(O.adaln(x, z, z, 1e-6), want, rtol=1e-10, atol=1e-10)


def test_adaln_shift_and_one_plus_scale():
    x = RNG.standard_normal((3, 64))
    sc = RNG.standard_normal((1, 64))
    sh = RNG.standard_normal((1, 64))
    ln = torch.nn.functional.layer_norm(torch.from_numpy(x), (64,), eps=1e-6).numpy()
    # scale = -1 kills the normalised term entirely, leaving the shift
    np.testing.assert_allclose(O.adaln(x, sh, -np.ones((1, 64)), 1e-6), np.broadcast_to(sh, x.shape), atol=1e-12)
    # linear in the shift, affine in the scale with slope LN(x)
    np.testing.assert_allclose(O.adaln(x, sh, sc, 1e-6) - O.adaln(x, 0 * sh, sc, 1e-6), np.broadcast_to(sh, x.shape), atol=1e-12)
    np.testing.assert_allclose(O.adaln(x, sh, sc + 1, 1e-6) - O.adaln(x, sh, sc, 1e-6), ln, atol=1e-10)


def test_rms_norm_against_library_and_constant_weight():
    x = RNG.standard_normal((5, 128)) * 4
    w = RNG.standard_normal(128)
    want = torch.nn.functional.rms_norm(torch.from_numpy(x), (128,), weight=torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rms_norm(x, w, 1e-6), want, rtol=1e-10, atol=1e-10)
    y = O.rms_norm(x, np.full(128, 2.5), 0.0)
    np.testing.assert_allclose(np.sqrt((y ** 2).mean(-1)), 2.5, rtol=1e-12)


def test_silu_and_swiglu():
    z = np.linspace(-30, 30, 601)
    want = torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    np.testing.assert_allclose(O.silu(z), want, rtol=1e-12, atol=1e-300)
    assert O.silu(np.array(0.0)) == 0.0
    g = RNG.standard_normal(10)
    # the first argument is the gated one: up = 1 leaves silu(gate)
    np.testing.assert_allclose(O.swiglu(g, np.ones(10)), O.silu(g))
    np.testing.assert_allclose(O.swiglu(np.full(10, 50.0), g), 50.0 * g)


# ------------------------------------------------------------------ attention
def _brute_attention(q, k, v):
    N, D = len(q), len(q[0])
    out = []
    for i in range(N):
        w = [math.exp(sum(q[i][d] * k[j][d] for d in range(D)) / math.sqrt(D)) for j in range(N)]
        tot = sum(w)
        out.append([sum(w[j] * v[j][d] for j in range(N)) / tot for d in range(D)])
    return out


def test_attention_brute_force_tiny():
    for N, D in ((1, 4), (5, 8), (9, 16)):
        q, k, v = (RNG.standard_normal((N, D)) for _ in range(3))
        got = O.attention(q[None, :, None], k[None, :, None], v[None, :, None])[0, :, 0]
        np.testing.assert_allclose(got, np.array(_brute_attention(q.tolist(), k.tolist(), v.tolist())), rtol=1e-12, atol=1e-12)


def test_attention_against_library_sdpa_and_heads_separate():
    q, k, v = (torch.randn(2, 3, 37, 128, dtype=torch.float64) for _ in range(3))
    want = torch.nn.functional.scaled_dot_product_attention(q, k, v).numpy()    # [B, h, N, D]
    got = O.attention(*(t.permute(0, 2, 1, 3).numpy() for t in (q, k, v)))     # [B, N, h, D]
    np.testing.assert_allclose(got.transpose(0, 2, 1, 3), want, rtol=1e-10, atol=1e-10)


def test_attention_special_cases():
    N, D = 11, 128
    v = RNG.standard_normal((N, D))
    q = RNG.standard_normal((N, D))
    k = np.tile(RNG.standard_normal((1, D)), (N, 1))      # identical keys -> mean of V
    got = O.attention(q[None, :, None], k[None, :, None], v[None, :, None])[0, :, 0]
    np.testing.assert_allclose(got, np.broadcast_to(v.mean(0), got.shape), rtol=1e-12, atol=1e-12)
    k = np.zeros((N, D)); k[4] = 1e3 * q[0] / np.linalg.norm(q[0])  # one dominant logit
    got = O.attention(q[:1][None, :, None], k[None, :, None], v[None, :, None])[0, 0, 0]
    np.testing.assert_allclose(got, v[4], atol=1e-12)
    # large logits stay finite (row maximum subtracted)
    qq = RNG.standard_normal((N, D)) * 100
    assert np.isfinite(O.attention(qq[None, :, None], qq[None, :, None], v[None, :, None])).all()


# ------------------------------------------------------------------ timestep / modulation
def test_sinusoid_closed_forms():
    e = O.timestep_sinusoid(np.array([0.0]), 256)
    np.testing.assert_array_equal(e, np.concatenate([np.ones((1, 128)), np.zeros((1, 128))], 1))
    # sigma = 1e-3 -> tau = 1: element 0 is cos(1), element 128 is sin(1); the last
    # frequency is 10000^(-127/128)
    e = O.timestep_sinusoid(np.array([1e-3]), 256)
    assert abs(e[0, 0] - math.cos(1.0)) < 1e-15 and abs(e[0, 128] - math.sin(1.0)) < 1e-15
    assert abs(e[0, 255] - math.sin(10000.0 ** (-127.0 / 128.0))) < 1e-15


def test_modulation_slots_and_zero_input_path():
    cfg = O.Config.tiny()
    H = cfg.hidden
    w_in = RNG.standard_normal((H, 256)) * 0.02
    w_out = RNG.standard_normal((H, H)) * 0.02
    # W_mod picks slot s from a one-hot of e: every slot of m is silu(e) seen through it
    w_mod = np.zeros((17 * H, H))
    for s in range(17):
        w_mod[s * H:(s + 1) * H] = np.eye(H) * (s + 1)
    m = O.modulation(np.array([0.3, 0.7]), w_in, w_out, w_mod, cfg)
    parts = O.split_modulation(m, H)
    assert list(parts)[0] == "img_shift_a" and list(parts)[6] == "txt_shift_a"
    assert list(parts)[12] == "single_shift" and list(parts)[15] == "final_shift"
    base = parts["img_shift_a"][:, 0]
    for s, name in enumerate(parts):
        np.testing.assert_allclose(parts[name][:, 0], base * (s + 1), rtol=1e-12)
    # sigma enters only through the sinusoid: equal sigma -> equal rows
    m2 = O.modulation(np.array([0.5, 0.5]), w_in, w_out, w_mod, cfg)
    np.testing.assert_array_equal(m2[0], m2[1])


def test_modulation_closed_form_at_sigma_zero():
    """At sigma = 0 the sinusoid is [1 ... 1 | 0 ... 0].  With W_in putting c_r on the first
    cosine column of row r, W_out = I and W_mod = 17 stacked identities, every slot of m must
    be silu(silu(c)) (the library SiLU): pins both SiLUs of the timestep MLP and the one
    before the modulation projection."""
    cfg = O.Config.tiny()
    H = cfg.hidden
    c = np.linspace(-4.0, 4.0, H)
    w_in = np.zeros((H, 256))
    w_in[:, 0] = c
    w_mod = np.vstack([np.eye(H)] * 17)
    m = O.modulation(np.array([0.0]), w_in, np.eye(H), w_mod, cfg)
    silu = lambda t: torch.nn.functional.silu(torch.from_numpy(t)).numpy()
    want = np.tile(silu(silu(c)), 17)
    np.testing.assert_allclose(m[0], want, rtol=1e-12, atol=1e-15)


# ------------------------------------------------------------------ blocks
def _tiny_block_setup(seed=0, batch=1, n_txt=8, grid=(3, 4), ref=((2, 2),)):
    wd = synth.TINY
    wl = synth.Workload("t", wd, batch, n_txt, grid, ref)
    g = synth.generator(seed)
    img, txt = synth.stream_weights(wd, g), synth.stream_weights(wd, g)
    sgl = synth.single_weights(wd, g)
    bi = synth.block_inputs(wl, seed)
    cfg = Hx.oracle_config(wd)
    ids = O.token_ids(n_txt, grid[0], grid[1], ref)
    c, s = O.rope_table(ids, cfg.axes_dim, cfg.rope_theta)
    x = Hx.to_np(bi["x"])
    m = Hx.to_np(bi["mod"])
    return cfg, wl, Hx.oracle_stream(img), Hx.oracle_stream(txt), Hx.oracle_single(sgl), x, m, c, s


def test_dual_block_zero_gates_leave_residual_unchanged():
    cfg, wl, wi, wt, ws, x, m, c, s = _tiny_block_setup()
    H = cfg.hidden
    m[:, 2 * H:3 * H] = 0; m[:, 5 * H:6 * H] = 0; m[:, 8 * H:9 * H] = 0; m[:, 11 * H:12 * H] = 0
    y = O.dual_block(x, wl.n_txt, wi, wt, O.split_modulation(m, H), c, s, cfg)
    np.testing.assert_array_equal(y, x)


def test_dual_block_routes_streams_to_their_modulation():
    cfg, wl, wi, wt, ws, x, m, c, s = _tiny_block_setup()
    H = cfg.hidden
    m_img_off = m.copy(); m_img_off[:, 2 * H:3 * H] = 0; m_img_off[:, 5 * H:6 * H] = 0
    y = O.dual_block(x, wl.n_txt, wi, wt, O.split_modulation(m_img_off, H), c, s, cfg)
    np.testing.assert_array_equal(y[:, wl.n_txt:], x[:, wl.n_txt:])     # image + reference rows untouched
    assert np.abs(y[:, :wl.n_txt] - x[:, :wl.n_txt]).max() > 1e-3
    m_txt_off = m.copy(); m_txt_off[:, 8 * H:9 * H] = 0; m_txt_off[:, 11 * H:12 * H] = 0
    y = O.dual_block(x, wl.n_txt, wi, wt, O.split_modulation(m_txt_off, H), c, s, cfg)
    np.testing.assert_array_equal(y[:, :wl.n_txt], x[:, :wl.n_txt])
    assert np.abs(y[:, wl.n_txt:] - x[:, wl.n_txt:]).max() > 1e-3


def test_dual_block_attention_is_joint_and_streams_use_own_weights():
    cfg, wl, wi, wt, ws, x, m, c, s = _tiny_block_setup()
    mod = O.split_modulation(m, cfg.hidden)
    y = O.dual_block(x, wl.n_txt, wi, wt, mod, c, s, cfg)
    x2 = x.copy(); x2[:, -1] += RNG.standard_normal(x.shape[-1])  # perturb one reference row (not by a constant: LN removes that)
    y2 = O.dual_block(x2, wl.n_txt, wi, wt, mod, c, s, cfg)
    assert np.abs(y2[:, 0] - y[:, 0]).max() > 1e-6                     # text row sees it
    # swapping the text weights changes only... everything (joint attention), but the
    # image rows' MLP uses the image weights: zero image MLP-out -> image rows differ from txt-MLP-zeroed run
    wi0 = O.StreamWeights(**{**wi.__dict__, "mlp_out": np.zeros_like(wi.mlp_out)})
    y3 = O.dual_block(x, wl.n_txt, wi0, wt, mod, c, s, cfg)
    np.testing.assert_array_equal(y3[:, :wl.n_txt], y[:, :wl.n_txt])
    assert np.abs(y3[:, wl.n_txt:] - y[:, wl.n_txt:]).max() > 1e-4


def test_single_block_zero_gate_and_permutation_equivariance():
    cfg, wl, wi, wt, ws, x, m, c, s = _tiny_block_setup(ref=())
    H = cfg.hidden
    m0 = m.copy(); m0[:, 14 * H:15 * H] = 0
    np.testing.assert_array_equal(O.single_block(x, ws, O.split_modulation(m0, H), c, s, cfg), x)
    # with every id equal, RoPE is one rotation for all rows: permuting rows permutes outputs
    ids = np.zeros((x.shape[1], 4)); ids[:, 1] = 5
    c1, s1 = O.rope_table(ids)
    mod = O.split_modulation(m, H)
    perm = RNG.permutation(x.shape[1])
    y = O.single_block(x, ws, mod, c1, s1, cfg)
    yp = O.single_block(x[:, perm], ws, mod, c1, s1, cfg)
    np.testing.assert_allclose(yp, y[:, perm], rtol=1e-10, atol=1e-10)


def _layer_norm_textbook(x, eps=1e-6):
    mu = x.mean(-1, keepdims=True)
    return (x - mu) / np.sqrt(((x - mu) ** 2).mean(-1, keepdims=True) + eps)


def _permutation(n, rng):
    """A permutation p with p != p^-1, and the [out, in] matrix P of the map o -> o[p]."""
    while True:
        p = rng.permutation(n)
        if (p != np.argsort(p)).any():
            break
    P = np.zeros((n, n))
    P[np.arange(n), p] = 1.0
    return p, P


def test_dual_block_uniform_attention_closed_form():
    """Zero q and k rows make every score 0, so attention is the mean of V over all N joint
    rows (both streams); with out = a permutation matrix, zero MLP-out and zero shift/scale,
    each row must be x + gate_a * o[p].  Pins the V slice of the qkv weight, joint attention,
    each stream's gate slot and own weights, and the [out, in] orientation of a square
    projection (y W^T: a transposed W gives o[p^-1])."""
    cfg, wl, wi, wt, ws, x, m, c, s = _tiny_block_setup()
    H, n_txt = cfg.hidden, wl.n_txt
    rng = np.random.default_rng(11)
    (p_i, P_i), (p_t, P_t) = _permutation(H, rng), _permutation(H, rng)

    def prep(w, P):
        qkv = w.qkv.copy()
        qkv[:2 * H] = 0
        return O.StreamWeights(**{**w.__dict__, "qkv": qkv, "out": P, "mlp_out": np.zeros_like(w.mlp_out)})

    m2 = m.copy()
    m2[:, 0:2 * H] = 0          # image stream shift_a, scale_a
    m2[:, 6 * H:8 * H] = 0      # text stream shift_a, scale_a
    y = O.dual_block(x, n_txt, prep(wi, P_i), prep(wt, P_t), O.split_modulation(m2, H), c, s, cfg)
    ln = _layer_norm_textbook(x)
    v = np.concatenate([ln[:, :n_txt] @ wt.qkv[2 * H:].T, ln[:, n_txt:] @ wi.qkv[2 * H:].T], axis=1)
    o = v.mean(axis=1, keepdims=True)
    want_t = x[:, :n_txt] + m[:, None, 8 * H:9 * H] * o[..., p_t]
    want_i = x[:, n_txt:] + m[:, None, 2 * H:3 * H] * o[..., p_i]
    np.testing.assert_allclose(y[:, :n_txt], want_t, rtol=0, atol=1e-12)
    np.testing.assert_allclose(y[:, n_txt:], want_i, rtol=0, atol=1e-12)


def test_single_block_uniform_attention_closed_form():
    """The single-stream block under the same construction: q, k and MLP-gate rows of the
    fused projection zero (silu(0) = 0, so act = 0 whatever the up rows), the attention part
    of out a permutation: x + gate * o[p].  Pins the column order [q | k | v | gate | up] of
    the fused projection and the [attn | act] order and orientation of the out-projection."""
    cfg, wl, wi, wt, ws, x, m, c, s = _tiny_block_setup(ref=())
    H, F = cfg.hidden, cfg.mlp_hidden
    p, P = _permutation(H, np.random.default_rng(12))
    qkv_mlp = ws.qkv_mlp.copy()
    qkv_mlp[:2 * H] = 0
    qkv_mlp[3 * H:3 * H + F] = 0
    out = ws.out.copy()
    out[:, :H] = P
    ws2 = O.SingleWeights(**{**ws.__dict__, "qkv_mlp": qkv_mlp, "out": out})
    m2 = m.copy()
    m2[:, 12 * H:14 * H] = 0
    y = O.single_block(x, ws2, O.split_modulation(m2, H), c, s, cfg)
    o = (_layer_norm_textbook(x) @ ws.qkv_mlp[2 * H:3 * H].T).mean(axis=1, keepdims=True)
    np.testing.assert_allclose(y, x + m[:, None, 14 * H:15 * H] * o[..., p], rtol=0, atol=1e-12)


def test_blocks_mlp_gate_is_the_first_half():
    """Reading R9 (first half of the MLP-in rows is the gate): with coordinate 0 of every row
    12 above the rest, LN puts it near +9, so gate rows -10 e_0 give silu(< -60) < 1e-24 and
    the MLP adds nothing, whatever the up rows; the same rows in the up half leave the MLP on.
    V rows are zeroed so the attention adds nothing either."""
    cfg, wl, wi, wt, ws, x, m, c, s = _tiny_block_setup()
    H, F, n_txt = cfg.hidden, cfg.mlp_hidden, wl.n_txt
    x2 = x.copy()
    x2[..., 0] += 12.0
    assert _layer_norm_textbook(x2)[..., 0].min() > 6.0

    def dual_w(w, off_half):
        qkv = w.qkv.copy()
        qkv[2 * H:] = 0
        mi = w.mlp_in.copy()
        rows = slice(0, F) if off_half == "gate" else slice(F, 2 * F)
        mi[rows] = 0
        mi[rows, 0] = -10.0
        return O.StreamWeights(**{**w.__dict__, "qkv": qkv, "mlp_in": mi})

    mod = O.split_modulation(m, H)
    y = O.dual_block(x2, n_txt, dual_w(wi, "gate"), dual_w(wt, "gate"), mod, c, s, cfg)
    np.testing.assert_allclose(y, x2, rtol=0, atol=1e-20)
    y_up = O.dual_block(x2, n_txt, dual_w(wi, "up"), dual_w(wt, "up"), mod, c, s, cfg)
    assert np.abs(y_up - x2).max() > 1e-2

    cfg1, wl1, _, _, ws1, x1, m1, c1, s1 = _tiny_block_setup(ref=())
    x1[..., 0] += 12.0

    def single_w(off_half):
        w = ws1.qkv_mlp.copy()
        w[2 * H:3 * H] = 0
        rows = slice(3 * H, 3 * H + F) if off_half == "gate" else slice(3 * H + F, 3 * H + 2 * F)
        w[rows] = 0
        w[rows, 0] = -10.0
        return O.SingleWeights(**{**ws1.__dict__, "qkv_mlp": w})

    mod1 = O.split_modulation(m1, H)
    np.testing.assert_allclose(O.single_block(x1, single_w("gate"), mod1, c1, s1, cfg1), x1, rtol=0, atol=1e-20)
    assert np.abs(O.single_block(x1, single_w("up"), mod1, c1, s1, cfg1) - x1).max() > 1e-2


def test_dual_block_mlp_uses_its_own_modulation_slots():
    """With the V rows zeroed the attention adds nothing, so the attention's shift and scale
    (slots 0, 1, 6, 7) must not change the output at all, a zero MLP gate (slots 5, 11) must
    leave x unchanged, and the MLP's shift (slots 3, 9) must matter."""
    cfg, wl, wi, wt, ws, x, m, c, s = _tiny_block_setup()
    H, n_txt = cfg.hidden, wl.n_txt

    def no_v(w):
        qkv = w.qkv.copy()
        qkv[2 * H:] = 0
        return O.StreamWeights(**{**w.__dict__, "qkv": qkv})

    wi0, wt0 = no_v(wi), no_v(wt)
    run = lambda mm: O.dual_block(x, n_txt, wi0, wt0, O.split_modulation(mm, H), c, s, cfg)
    y = run(m)
    m_a = m.copy()
    for slot in (0, 1, 6, 7):
        m_a[:, slot * H:(slot + 1) * H] += RNG.standard_normal((m.shape[0], H))
    np.testing.assert_array_equal(run(m_a), y)
    m_g = m.copy()
    m_g[:, 5 * H:6 * H] = 0
    m_g[:, 11 * H:12 * H] = 0
    np.testing.assert_array_equal(run(m_g), x)
    m_s = m.copy()
    m_s[:, 3 * H:4 * H] += 1.0
    m_s[:, 9 * H:10 * H] += 1.0
    assert np.abs(run(m_s)[:, :n_txt] - y[:, :n_txt]).max() > 1e-4
    assert np.abs(run(m_s)[:, n_txt:] - y[:, n_txt:]).max() > 1e-4


def test_dual_and_single_blocks_agree_on_the_attention_path():
    """The two block forms compute the same attention sub-layer by separate code: a dual
    block whose streams share one weight set and one modulation, with its MLP off (zero
    MLP-out), must equal a single block with the same q/k/v/out weights and norm weights,
    its MLP off (zero gate rows: act = silu(0) up = 0).  A slip in either path's q/k
    handling (norm order, a swapped norm weight, RoPE missing or on one operand) breaks
    the agreement; the shared helpers have their own pins."""
    cfg, wl, wi, wt, ws, x, m, c, s = _tiny_block_setup()
    H, F = cfg.hidden, cfg.mlp_hidden
    sw = O.StreamWeights(qkv=ws.qkv_mlp[:3 * H].copy(), q_norm=ws.q_norm, k_norm=ws.k_norm,
                         out=ws.out[:, :H].copy(), mlp_in=wi.mlp_in, mlp_out=np.zeros_like(wi.mlp_out))
    m2 = m.copy()
    for stream0 in (0, 6):                    # both streams' attention slots = the single slots
        m2[:, stream0 * H:(stream0 + 3) * H] = m[:, 12 * H:15 * H]
    qkv_mlp = ws.qkv_mlp.copy()
    qkv_mlp[3 * H:3 * H + F] = 0
    ws0 = O.SingleWeights(**{**ws.__dict__, "qkv_mlp": qkv_mlp})
    mod = O.split_modulation(m2, H)
    y_dual = O.dual_block(x, wl.n_txt, sw, sw, mod, c, s, cfg)
    y_single = O.single_block(x, ws0, mod, c, s, cfg)
    np.testing.assert_allclose(y_dual, y_single, rtol=0, atol=1e-12)
    assert np.abs(y_single - x).max() > 1e-3   # the attention sub-layer is not trivial here


def test_blocks_batch_rows_independent():
    cfg, wl, wi, wt, ws, x, m, c, s = _tiny_block_setup(batch=3)
    mod = O.split_modulation(m, cfg.hidden)
    y = O.dual_block(x, wl.n_txt, wi, wt, mod, c, s, cfg)
    y1 = O.dual_block(x[1:2], wl.n_txt, wi, wt, O.split_modulation(m[1:2], cfg.hidden), c, s, cfg)
    np.testing.assert_allclose(y[1:2], y1, rtol=1e-13, atol=1e-13)
    z = O.single_block(x, ws, mod, c, s, cfg)
    z1 = O.single_block(x[2:3], ws, O.split_modulation(m[2:3], cfg.hidden), c, s, cfg)
    np.testing.assert_allclose(z[2:3], z1, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ whole step / loop
def _tiny_step():
    wd = synth.TINY
    wl = synth.Workload("t", wd, 2, 16, (4, 4), ((2, 3),))
    w = synth.model_weights(wd, seed=5)
    inp = synth.step_inputs(wl, seed=5)
    ids = O.token_ids(wl.n_txt, *wl.grid, wl.ref_grids)
    return wd, wl, w, inp, ids


def test_step_fp32_agrees_with_fp64():
    wd, wl, w, inp, ids = _tiny_step()
    args = [Hx.to_np(inp["img_tokens"]), Hx.to_np(inp["ref_tokens"]), Hx.to_np(inp["txt_emb"]),
            Hx.to_np(inp["sigma"]), ids]
    v64 = O.dit_step(Hx.oracle_weights(wd, w, np.float64), *args, dtype=np.float64)
    v32 = O.dit_step(Hx.oracle_weights(wd, w, np.float32), *[a.astype(np.float32) if a.dtype != np.int32 else a for a in args], dtype=np.float32)
    assert v64.shape == (2, 16, 128)
    assert Hx.cosine(v32, v64) > 0.99999


def test_step_uses_only_target_rows_and_ref_tokens_matter():
    wd, wl, w, inp, ids = _tiny_step()
    ow = Hx.oracle_weights(wd, w)
    a = [Hx.to_np(inp["img_tokens"]), Hx.to_np(inp["ref_tokens"]), Hx.to_np(inp["txt_emb"]), Hx.to_np(inp["sigma"]), ids]
    v = O.dit_step(ow, *a)
    a2 = list(a); a2[1] = a[1] + 1.0
    v2 = O.dit_step(ow, *a2)
    assert v.shape == v2.shape and np.abs(v - v2).max() > 1e-6


def test_step_without_blocks_maps_each_target_token_to_its_own_velocity_row():
    """With no blocks, nothing mixes rows: the text features must not touch the velocity,
    and changing image token j must change velocity row j only (the final layer reads the
    target rows, which follow the text rows)."""
    wd, wl, w, inp, ids = _tiny_step()
    ow = Hx.oracle_weights(wd, w)
    img, ref, txt = Hx.to_np(inp["img_tokens"]), Hx.to_np(inp["ref_tokens"]), Hx.to_np(inp["txt_emb"])
    sig = Hx.to_np(inp["sigma"])
    step = lambda i, t: O.dit_step(ow, i, ref, t, sig, ids, n_dual=0, n_single=0)
    v = step(img, txt)
    np.testing.assert_array_equal(step(img, txt + 1.0), v)
    j = 5
    img2 = img.copy()
    img2[:, j] += RNG.standard_normal(img.shape[-1])
    d = np.abs(step(img2, txt) - v).max(axis=-1)
    assert (d[:, j] > 1e-6).all()
    assert (np.delete(d, j, axis=1) == 0).all()
    # the final layer normalises: scaling every target token by 3 scales each embedded row
    # by 3, which LayerNorm removes (up to its eps against a row variance of ~0.05)
    np.testing.assert_allclose(step(3.0 * img, txt), v, rtol=1e-3, atol=1e-4)


def test_euler_loop_telescopes_and_schedule_ends_at_zero():
    sig = O.sigma_schedule(0.8, int(STRUCT["steps"]))
    assert len(sig) == 5 and sig[0] == 0.8 and sig[-1] == 0.0
    # reading R19's interior, in closed form: equal steps of sigma_0 / 4 (no time shift)
    np.testing.assert_allclose(sig, [0.8, 0.6, 0.4, 0.2, 0.0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(O.sigma_schedule(1.0, 4), [1.0, 0.75, 0.5, 0.25, 0.0], rtol=0, atol=0)
    x = RNG.standard_normal((2, 3))
    v = RNG.standard_normal((2, 3))
    y = x
    for k in range(4):
        y = O.euler_update(y, v, sig[k], sig[k + 1])
    np.testing.assert_allclose(y, x - 0.8 * v, rtol=1e-13, atol=1e-13)


def test_klein_parameter_count_is_about_4b():
    # no biases anywhere (reading R17) gives the card's "4B" at klein width
    w = synth.model_weights(synth.KLEIN, seed=0, device="meta")
    n = sum(t.numel() for t in [w["mod"]["t_in"], w["mod"]["t_out"], w["mod"]["mod"], w["x_emb"], w["ctx_emb"], w["proj_out"]])
    n += sum(t.numel() for a, b in w["dual"] for t in list(a.values()) + list(b.values()))
    n += sum(t.numel() for s in w["single"] for t in s.values())
    billions = n / 1e9
    assert abs(billions - float(STRUCT["model_params_billion"])) < 0.25, billions
    assert len(w["dual"]) == int(STRUCT["n_dual"]) and len(w["single"]) == int(STRUCT["n_single"])
    assert synth.KLEIN.txt_dim == int(STRUCT["text_dim"]) == 3 * 2560


# ---- e4m3 quantisation (reading R26): pinned by encodings fixed by the format's definition
def test_e4m3_known_encodings_ties_and_saturation():
    # 1 = 2^0 (e 7, m 0); 448 = 2^8 * 1.75 (e 15, m 6); 240 = 2^7 * 1.875 (e 14, m 7);
    # 2^-6 is the smallest normal (e 1); 2^-9 the smallest subnormal (m 1); -2 = sign | e 8
    fixed = {1.0: 0x38, 448.0: 0x7E, 240.0: 0x77, 2.0 ** -6: 0x08, 2.0 ** -9: 0x01, -2.0: 0xC0, 0.0: 0x00,
             0.3125: 0x2A}
    for v, code in fixed.items():
        assert O.e4m3_encode(v) == code, (v, hex(O.e4m3_encode(v)))
    # ties go to the even mantissa: 1.0625 between m 0 and m 1 -> m 0; 1.1875 between m 1 and
    # m 2 -> m 2; 2^-10 between 0 and the smallest subnormal -> 0
    assert O.e4m3_encode(1.0625) == 0x38 and O.e4m3_encode(1.1875) == 0x3A and O.e4m3_encode(2.0 ** -10) == 0x00
    # nearest, not truncation: 0.3 lies nearer 0.3125 (m 2) than 0.28125 (m 1)
    assert O.e4m3_encode(0.3) == 0x2A
    # saturation to the largest finite value instead of NaN / overflow
    assert O.e4m3_encode(464.0) == 0x7E and O.e4m3_encode(1e9) == 0x7E and O.e4m3_encode(-1e9) == 0xFE
    assert O.e4m3_encode(470.0) == 0x7E and O.e4m3_encode(-447.0) == 0xFE
    # zero keeps its sign, as in the IEEE formats: -0 and negative values that round to
    # zero give the negative-zero code
    assert O.e4m3_encode(-0.0) == 0x80 and O.e4m3_encode(-1e-6) == 0x80 and O.e4m3_encode(1e-6) == 0x00


def test_e4m3_codes_round_trip_and_are_monotonic():
    finite = [c for c in range(128) if c != 0x7F]
    vals = [O.e4m3_decode(c) for c in finite]
    assert all(b > a for a, b in zip(vals, vals[1:]))                 # strictly increasing magnitudes
    assert vals[-1] == 448.0 and vals[1] == 2.0 ** -9
    for c in finite + [c | 0x80 for c in finite if c]:
        assert O.e4m3_encode(O.e4m3_decode(c)) == c
    assert np.isnan(O.e4m3_decode(0x7F)) and np.isnan(O.e4m3_decode(0xFF))


def test_quantize_rows_e4m3_scales_and_zero_rows():
    w = np.zeros((3, 16), np.float32)
    w[0, 5] = -896.0          # max |w| = 896 -> scale 2, the element maps to -448
    w[0, 6] = 1.0             # 1 / 2 = 0.5 -> e 6, m 0
    w[2] = 0.25
    codes, scale = O.quantize_rows_e4m3(w)
    assert scale.tolist() == [2.0, 1.0, np.float32(0.25 / 448.0)]
    assert codes[0, 5] == 0xFE and codes[0, 6] == 0x30 and codes[0, 0] == 0x00
    assert (codes[1] == 0).all()                                      # all-zero row: scale 1, codes 0
    assert (codes[2] == 0x7E).all()                                   # the row maximum maps to 448


# ---- the e4m3 variant's arithmetic (reading R26): the vectorised quantiser is pinned to
# the scalar, definition-pinned encoder above; the quantised linear to brute force and to
# exact cases; the blocks to the list of projections the variant names
def _e4m3_finite_values():
    return np.array(sorted({O.e4m3_decode(c) for c in range(256) if c not in (0x7F, 0xFF)}))


def test_e4m3_round_matches_the_scalar_encoder_everywhere():
    v = _e4m3_finite_values()
    mid = 0.5 * (v[1:] + v[:-1])
    rng = np.random.default_rng(7)
    wide = rng.standard_normal(50000) * np.exp(rng.uniform(-14.0, 7.0, 50000))
    xs = np.concatenate([v, mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf), wide,
                         [448.0, 460.0, 464.0, 465.0, 1e30, -1e30, 2.0 ** -10, -2.0 ** -10, 0.0, -0.0]])
    xs = xs.astype(np.float32)
    got = O.e4m3_round(xs)
    want = np.array([O.e4m3_decode(O.e4m3_encode(float(x))) for x in xs])
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(np.signbit(got), np.signbit(want))     # -0 and small negatives keep the sign


def test_quantize_rows_values_match_the_codes():
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((40, 96)) * np.exp(rng.uniform(-6, 6, (40, 1)))).astype(np.float32)
    x[5] = 0.0
    x[7, 3] = 1e6
    codes, scale = O.quantize_rows_e4m3(x)
    vals, scale2 = O.quantize_rows_e4m3_values(x)
    np.testing.assert_array_equal(scale2, scale)
    np.testing.assert_array_equal(vals, np.vectorize(O.e4m3_decode)(codes))
    # leading axes are rows too: a [2, 20, 96] array is quantised like its 40 rows
    v3, s3 = O.quantize_rows_e4m3_values(x.reshape(2, 20, 96))
    np.testing.assert_array_equal(v3.reshape(40, 96), vals)
    np.testing.assert_array_equal(s3.reshape(40), scale)


def test_bf16_round_matches_the_library_conversion_and_ties():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(O.bf16_round(x), lib)
    # ties to even: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 (kept mantissa even: 1);
    # 1 + 3 2^-8 halfway between 1 + 2^-7 and 1 + 2^-6 (even: 1 + 2^-6); negatives mirror
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), -(1 + 3 * 2.0 ** -8)], np.float32)
    np.testing.assert_array_equal(O.bf16_round(ties), [1.0, 1 + 2.0 ** -6, -1.0, -(1 + 2.0 ** -6)])
    assert O.bf16_round(np.float32(1 + 2.0 ** -7)) == np.float32(1 + 2.0 ** -7)   # already bf16: unchanged


def test_linear_e4m3_brute_force_and_exact_cases():
    rng = np.random.default_rng(10)
    a = rng.standard_normal((3, 5, 32)).astype(np.float32) * np.float32(1.7)
    w = (rng.standard_normal((6, 32)) * 0.05).astype(np.float32)
    got = O.linear_e4m3(a, w)
    # brute force from the scalar, definition-pinned quantiser: sum over k of the decoded
    # codes' products, times the token row's scale and the output row's scale
    ca, sa = O.quantize_rows_e4m3(a.reshape(15, 32))
    cw, sw = O.quantize_rows_e4m3(w)
    dec = np.vectorize(O.e4m3_decode)
    want = np.zeros((15, 6))
    for m in range(15):
        for n in range(6):
            want[m, n] = sum(dec(ca[m, k]) * dec(cw[n, k]) for k in range(32)) * float(sa[m]) * float(sw[n])
    np.testing.assert_allclose(got.reshape(15, 6), want, rtol=1e-12, atol=1e-15)
    # rows that already lie on the grid (every element an e4m3 value times a power of two,
    # the row maximum 448 times it) are quantised without loss: the product is exact
    grid = _e4m3_finite_values()
    ga = rng.choice(grid, (4, 16)); ga[:, 0] = 448.0
    gw = rng.choice(grid, (3, 16)); gw[:, 3] = -448.0
    ga, gw = ga * 2.0 ** -5, gw * 2.0 ** -12
    np.testing.assert_allclose(O.linear_e4m3(ga, gw), ga @ gw.T, rtol=1e-14, atol=0)
    # a token row's scale and an output row's scale act on their own row / column only:
    # scaling token row 1 of a by 2^3 scales output row 1 by 2^3 exactly
    a2 = a.reshape(15, 32).copy(); a2[1] *= 8.0
    g2 = O.linear_e4m3(a2, w)
    np.testing.assert_array_equal(g2[1], 8.0 * got.reshape(15, 6)[1])
    np.testing.assert_array_equal(np.delete(g2, 1, 0), np.delete(got.reshape(15, 6), 1, 0))
    w2 = w.copy(); w2[4] *= 0.25
    g3 = O.linear_e4m3(a, w2)
    np.testing.assert_array_equal(g3[..., 4], 0.25 * got[..., 4])
    np.testing.assert_array_equal(np.delete(g3, 4, -1), np.delete(got, 4, -1))


def _recording_quantiser(monkeypatch, identity=False):
    """Replace the per-row quantiser by a recorder of its inputs (identity=True: also
    pass the input through unquantised, with unit scales)."""
    seen = []
    real = O.quantize_rows_e4m3_values

    def rec(x):
        x32 = np.asarray(x, np.float32)
        seen.append((x32.shape, bool((O.bf16_round(x32) == x32).all())))
        if identity:
            return np.asarray(x, np.float64), np.ones(x32.shape[:-1], np.float32)
        return real(x)

    monkeypatch.setattr(O, "quantize_rows_e4m3_values", rec)
    return seen


def test_e4m3_blocks_quantise_the_projections_the_variant_names(monkeypatch):
    cfg, wl, wi, wt, ws, x, m, c, s = _tiny_block_setup()
    H, F, N = cfg.hidden, cfg.mlp_hidden, x.shape[1]
    nt, ni = wl.n_txt, N - wl.n_txt
    mod = O.split_modulation(m, H)
    # with the quantiser replaced by the identity (and every stored value already bf16,
    # which the identity path cannot see), the e4m3 blocks are the plain blocks: the variant
    # changes nothing but the quantised projections
    seen = _recording_quantiser(monkeypatch, identity=True)
    monkeypatch.setattr(O, "bf16_round", lambda a: np.asarray(a))
    np.testing.assert_allclose(O.dual_block(x, nt, wi, wt, mod, c, s, cfg, e4m3="all"),
                               O.dual_block(x, nt, wi, wt, mod, c, s, cfg), rtol=0, atol=1e-12)
    np.testing.assert_allclose(O.single_block(x, ws, mod, c, s, cfg, e4m3="all"),
                               O.single_block(x, ws, mod, c, s, cfg), rtol=0, atol=1e-12)
    monkeypatch.undo()
    # which operands are quantised, in order, and which ones the quantiser reads as stored
    # bf16 values (the attention output and the activations, reading R18) or unrounded
    # (the adaLN outputs, which the GPU quantises straight from fp32)
    seen = _recording_quantiser(monkeypatch)
    O.dual_block(x, nt, wi, wt, mod, c, s, cfg, e4m3="all")
    shapes = [sh for sh, _ in seen]
    per_stream = lambda n: [(1, n, H), (3 * H, H)]
    assert shapes == (per_stream(nt) + per_stream(ni) +                       # QKV: txt, img
                      [(1, nt, H), (H, H), (1, nt, H), (2 * F, H), (1, nt, F), (H, F)] +   # txt: out, MLP-in, MLP-out
                      [(1, ni, H), (H, H), (1, ni, H), (2 * F, H), (1, ni, F), (H, F)]), shapes
    stored = [b for (sh, b), i in zip(seen, range(len(seen))) if i % 2 == 0]   # activations only
    assert stored == [False, False, True, False, True, True, False, True], stored
    seen.clear()
    O.single_block(x, ws, mod, c, s, cfg, e4m3="fused")
    assert [sh for sh, _ in seen] == [(1, N, H), (3 * H + 2 * F, H)] and not seen[0][1]
    seen.clear()
    O.single_block(x, ws, mod, c, s, cfg, e4m3="all")
    assert [sh for sh, _ in seen] == [(1, N, H), (3 * H + 2 * F, H), (1, N, H + F), (H, H + F)]
    assert seen[2][1] and not seen[0][1]
    # and e4m3=None quantises nothing
    seen.clear()
    O.dual_block(x, nt, wi, wt, mod, c, s, cfg)
    O.single_block(x, ws, mod, c, s, cfg)
    assert seen == []
