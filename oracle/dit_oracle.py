"""Oracle: a plain, slow CPU statement of one FLUX.2 [klein]-style DiT denoising step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or runs this
module: only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may.  It shares no code with the CUDA library (no kernels, headers,
helpers, tables or constant generators); both sides only consume the same seeded
inputs, which come from ``diffusion_transformer_step_gb300.synth``.

Every function is the definition written out in numpy, in float64 unless the caller
asks for float32, with no blocking, fusion or reordering beyond what the definition
states.  Inputs are the bf16-rounded weights and activations the GPU also sees,
upcast; no intermediate value is rounded, except in the e4m3 variant (reading R26),
whose quantisers take their rounding decisions on the values the GPU path feeds them.

Sources, cited by page title and section:
  [card]   "flux2-klein-p100a" model card (FLUX.2 [klein] 4B on one p100a):
           the Quickstart task table, Caveats.
  [pyref]  "tt_flux2_klein -- Python reference": Lower-level entry points, Modules,
           "Things that are easy to get wrong".
  [mstar]  "FLUX.2 [klein] 4B/9B + Z-Image-Turbo on a shared DiT scaffold": What does
           this PR do (batch rows independent bit for bit).
The pages name the blocks (5 dual-stream + 20 single-stream, the [pyref] Modules table)
but never write their maths out; every point they leave open is taken in its plainest
reading, labelled "reading Rn" below and listed with its basis in the design notes.

Parity status: every function here is pinned by tests/test_oracle_pins.py against
closed forms, library routines, invariants or brute force, except where a docstring
says "parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


# ----------------------------------------------------------------------------------
# Configuration
# ----------------------------------------------------------------------------------
@dataclass(frozen=True)
class Config:
    """Model widths.  ``klein()`` gives the 4B widths; the pages fix theta 2000,
    32 dims per RoPE axis ([pyref] "Things that are easy to get wrong"), a 7680-wide
    text feature (three 2560-wide encoder layers, [pyref] Lower-level entry points:
    encode) and 5 + 20 blocks ([pyref] Modules: tt_dit.py)."""
    hidden: int = 3072
    heads: int = 24
    head_dim: int = 128
    mlp_hidden: int = 9216
    n_dual: int = 5
    n_single: int = 20
    in_channels: int = 128
    txt_dim: int = 7680
    rope_theta: float = 2000.0
    axes_dim: tuple = (32, 32, 32, 32)
    eps: float = 1e-6           # reading R3: LayerNorm / RMSNorm epsilon
    time_dim: int = 256         # reading R13: sinusoid width
    time_max_period: float = 10000.0  # reading R13

    @staticmethod
    def klein() -> "Config":
        return Config()

    @staticmethod
    def tiny() -> "Config":
        return Config(hidden=256, heads=2, head_dim=128, mlp_hidden=768, n_dual=1, n_single=1)


# ----------------------------------------------------------------------------------
# Token ids and RoPE  ([pyref] "Things that are easy to get wrong"; readings R10-R12, R7)
# ----------------------------------------------------------------------------------
def token_ids(n_txt: int, grid_h: int, grid_w: int, ref_grids=()) -> np.ndarray:
    """(t, h, w, l) position ids of the joint sequence [text | target image | refs].

    Reading R10: text row i is (0, 0, 0, i); every padded row continues the count.
    Reading R11: target token (r, c) of the gh x gw patch grid, row-major, is (0, r, c, 0).
    [pyref]: reference image i gets t = 10 + 10*i; reading R12: over its own grid
    (r, c), row-major, l = 0.
    """
    rows = []
    for i in range(n_txt):
        rows.append((0, 0, 0, i))
    for r in range(grid_h):
        for c in range(grid_w):
            rows.append((0, r, c, 0))
    for i, (gh, gw) in enumerate(ref_grids):
        t = 10 + 10 * i
        for r in range(gh):
            for c in range(gw):
                rows.append((t, r, c, 0))
    return np.asarray(rows, dtype=np.int32).reshape(-1, 4)


def rope_angles(ids: np.ndarray, axes_dim=(32, 32, 32, 32), theta: float = 2000.0) -> np.ndarray:
    """Rotation angle of every adjacent pair, [N, sum(axes_dim)/2], float64.

    Reading R7: axis a owns dims [32a, 32a+32) of a head; its pair j = 0..15 is the
    adjacent dims (2j, 2j+1) of that slice ("repeat_interleave_real=True"), turned by
    pos_a * theta**(-2j/dim_a).
    """
    ids = np.asarray(ids, dtype=np.float64)
    cols = []
    for a, dim in enumerate(axes_dim):
        j = np.arange(dim // 2, dtype=np.float64)
        omega = theta ** (-(2.0 * j) / dim)
        cols.append(ids[:, a:a + 1] * omega[None, :])
    return np.concatenate(cols, axis=1)


def rope_table(ids: np.ndarray, axes_dim=(32, 32, 32, 32), theta: float = 2000.0):
    """cos and sin of every pair angle, each [N, head_dim/2], float64."""
    ang = rope_angles(ids, axes_dim, theta)
    return np.cos(ang), np.sin(ang)


def apply_rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate adjacent pairs of the last axis.  x: [..., N, heads, D]; cos/sin [N, D/2].

    For pair (x0, x1) = (x[2j], x[2j+1]): x0' = x0 cos - x1 sin, x1' = x0 sin + x1 cos.
    """
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    c = cos[:, None, :]
    s = sin[:, None, :]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


# ----------------------------------------------------------------------------------
# Norms and activations (readings R3-R5, R9)
# ----------------------------------------------------------------------------------
def layer_norm(x: np.ndarray, eps: float) -> np.ndarray:
    """LayerNorm over the last axis, no affine, biased variance (reading R3)."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def adaln(x: np.ndarray, shift: np.ndarray, scale: np.ndarray, eps: float) -> np.ndarray:
    """Adaptive LayerNorm: (1 + scale) * LN(x) + shift (reading R4).
    shift/scale broadcast against x's last axis (shape [B, 1, H] for per-row-batch)."""
    return (1.0 + scale) * layer_norm(x, eps) + shift


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis with a learned weight (reading R5)."""
    ms = (x ** 2).mean(axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """Reading R9: the first half of the MLP-in output is the gate: silu(gate) * up."""
    return silu(gate) * up


# ----------------------------------------------------------------------------------
# Attention (reading R6; [card] Caveats and [pyref]: all 512 padded text rows, no mask)
# ----------------------------------------------------------------------------------
def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_chunk: int = 2048) -> np.ndarray:
    """Non-causal softmax attention with no mask, per batch row and head.

    q, k, v: [B, N, heads, D].  Returns [B, N, heads, D].
    S = q k^T / sqrt(D) over every key; softmax with the row maximum subtracted; S V.
    Query rows are processed in chunks only to bound memory: each row's softmax is
    independent, so chunking changes no arithmetic.
    """
    B, N, Hh, D = q.shape
    scale = 1.0 / math.sqrt(D)
    out = np.empty((B, N, Hh, D), dtype=q.dtype)
    for b in range(B):
        for h in range(Hh):
            kh = k[b, :, h, :]
            vh = v[b, :, h, :]
            for r0 in range(0, N, q_chunk):
                s = (q[b, r0:r0 + q_chunk, h, :] @ kh.T) * scale
                s = s - s.max(axis=1, keepdims=True)
                p = np.exp(s)
                p = p / p.sum(axis=1, keepdims=True)
                out[b, r0:r0 + q_chunk, h, :] = p @ vh
    return out


# ----------------------------------------------------------------------------------
# Timestep embedding and the global modulation (readings R13, R14;
# [card] Caveats and [pyref]: modulation is global per step, not per block)
# ----------------------------------------------------------------------------------
def timestep_sinusoid(sigma: np.ndarray, dim: int = 256, max_period: float = 10000.0) -> np.ndarray:
    """[cos(tau f_k) | sin(tau f_k)], tau = 1000 sigma, f_k = max_period**(-k/(dim/2))."""
    sigma = np.asarray(sigma, dtype=np.float64)
    half = dim // 2
    k = np.arange(half, dtype=np.float64)
    f = max_period ** (-k / half)
    arg = (1000.0 * sigma)[:, None] * f[None, :]
    return np.concatenate([np.cos(arg), np.sin(arg)], axis=1)


MOD_SLOTS = 17  # 6 img-dual + 6 txt-dual + 3 single + 2 final, each `hidden` wide (R14)


def modulation(sigma, w_t_in, w_t_out, w_mod, cfg: Config, dtype=np.float64) -> np.ndarray:
    """m = W_mod SiLU(e), e = W_out SiLU(W_in sinusoid(1000 sigma)).  Returns [B, 17H].
    No biases (reading R17); no guidance embedding (guidance 1.0, [card] task table)."""
    emb = timestep_sinusoid(sigma, cfg.time_dim, cfg.time_max_period).astype(dtype)
    h1 = silu(emb @ w_t_in.astype(dtype).T)
    e = h1 @ w_t_out.astype(dtype).T
    return silu(e) @ w_mod.astype(dtype).T


def split_modulation(m: np.ndarray, hidden: int) -> dict:
    """Name the 17 slots of the modulation vector (reading R14).  Each is [B, 1, H]."""
    names = ["img_shift_a", "img_scale_a", "img_gate_a", "img_shift_m", "img_scale_m", "img_gate_m",
             "txt_shift_a", "txt_scale_a", "txt_gate_a", "txt_shift_m", "txt_scale_m", "txt_gate_m",
             "single_shift", "single_scale", "single_gate",
             "final_shift", "final_scale"]
    out = {}
    for i, n in enumerate(names):
        out[n] = m[:, None, i * hidden:(i + 1) * hidden]
    return out


# ----------------------------------------------------------------------------------
# Blocks
# ----------------------------------------------------------------------------------
@dataclass
class StreamWeights:
    """One stream of a dual-stream block (logical layouts, [out, in], no biases).
    mlp_in is [gate; up] stacked along the output axis (reading R9)."""
    qkv: np.ndarray       # [3H, H]
    q_norm: np.ndarray    # [D]
    k_norm: np.ndarray    # [D]
    out: np.ndarray       # [H, H]
    mlp_in: np.ndarray    # [2F, H]
    mlp_out: np.ndarray   # [H, F]


@dataclass
class SingleWeights:
    """A single-stream block: one fused projection with columns [q|k|v|gate|up]
    (reading R8) and one out-projection over [attn | act]."""
    qkv_mlp: np.ndarray   # [3H + 2F, H]
    q_norm: np.ndarray    # [D]
    k_norm: np.ndarray    # [D]
    out: np.ndarray       # [H, H + F]


def _heads(x: np.ndarray, heads: int, head_dim: int) -> np.ndarray:
    B, N, _ = x.shape
    return x.reshape(B, N, heads, head_dim)


def _qk_norm_rope(q, k, qn, kn, cos, sin, cfg: Config):
    """Per-head RMSNorm of q and k (reading R5), then RoPE on both (reading R7)."""
    q = rms_norm(_heads(q, cfg.heads, cfg.head_dim), qn, cfg.eps)
    k = rms_norm(_heads(k, cfg.heads, cfg.head_dim), kn, cfg.eps)
    return apply_rope(q, cos, sin), apply_rope(k, cos, sin)


def _project(a, w, quantised: bool, dtype, stored_bf16: bool = False):
    """a @ w^T, or with both operands in e4m3 (linear_e4m3) when `quantised`.  `stored_bf16`
    marks an input the GPU path holds as bf16 before its quantising pass (the attention
    output and the SwiGLU activations, reading R18): the quantiser then sees that bf16
    value (reading R26)."""
    if not quantised:
        return a @ w.astype(dtype).T
    return linear_e4m3(bf16_round(a) if stored_bf16 else a, w, dtype)


def dual_block(x, n_txt, w_img: StreamWeights, w_txt: StreamWeights, mod: dict, cos, sin,
               cfg: Config, dtype=np.float64, e4m3=None) -> np.ndarray:
    """One dual-stream block over x = [B, N, H] with rows [txt | img | ref].

    Rows [0, n_txt) use the text weights and text modulation; every later row (target
    image and reference tokens) uses the image weights and image modulation (reading R1).
    Attention is joint over all N rows (reading R2).  Residuals are gated with the raw
    gate vector (reading R4).  e4m3 = "all" runs the four projections of both streams in
    e4m3 (reading R26: the QKV and MLP-in inputs are the adaLN outputs, the out and
    MLP-out inputs the stored attention output and activations).
    """
    H, F = cfg.hidden, cfg.mlp_hidden
    q8 = e4m3 == "all"
    x = x.astype(dtype)
    cast = lambda a: a.astype(dtype)
    streams = [("txt", slice(0, n_txt), w_txt), ("img", slice(n_txt, x.shape[1]), w_img)]
    qs, ks, vs = [], [], []
    for name, rows, w in streams:
        y = adaln(x[:, rows], mod[f"{name}_shift_a"], mod[f"{name}_scale_a"], cfg.eps)
        qkv = _project(y, w.qkv, q8, dtype)
        q, k, v = qkv[..., :H], qkv[..., H:2 * H], qkv[..., 2 * H:]
        q = rms_norm(_heads(q, cfg.heads, cfg.head_dim), cast(w.q_norm), cfg.eps)
        k = rms_norm(_heads(k, cfg.heads, cfg.head_dim), cast(w.k_norm), cfg.eps)
        qs.append(q); ks.append(k); vs.append(_heads(v, cfg.heads, cfg.head_dim))
    q = apply_rope(np.concatenate(qs, axis=1), cos, sin)
    k = apply_rope(np.concatenate(ks, axis=1), cos, sin)
    v = np.concatenate(vs, axis=1)
    attn = attention(q, k, v).reshape(x.shape[0], x.shape[1], H)
    out = x.copy()
    for name, rows, w in streams:
        xs = out[:, rows] + mod[f"{name}_gate_a"] * _project(attn[:, rows], w.out, q8, dtype, stored_bf16=True)
        y = adaln(xs, mod[f"{name}_shift_m"], mod[f"{name}_scale_m"], cfg.eps)
        h = _project(y, w.mlp_in, q8, dtype)
        act = swiglu(h[..., :F], h[..., F:])
        out[:, rows] = xs + mod[f"{name}_gate_m"] * _project(act, w.mlp_out, q8, dtype, stored_bf16=True)
    return out


def single_block(x, w: SingleWeights, mod: dict, cos, sin, cfg: Config, dtype=np.float64,
                 e4m3=None) -> np.ndarray:
    """One single-stream block: one weight set over the joint sequence, attention and
    MLP in parallel from the same modulated input (reading R8).  e4m3 = "fused" runs the
    fused QKV + MLP-in projection in e4m3, "all" the out-projection over [attn | act] too
    (reading R26)."""
    H, F = cfg.hidden, cfg.mlp_hidden
    x = x.astype(dtype)
    y = adaln(x, mod["single_shift"], mod["single_scale"], cfg.eps)
    h = _project(y, w.qkv_mlp, e4m3 in ("fused", "all"), dtype)
    q, k, v = h[..., :H], h[..., H:2 * H], h[..., 2 * H:3 * H]
    gate, up = h[..., 3 * H:3 * H + F], h[..., 3 * H + F:]
    q, k = _qk_norm_rope(q, k, w.q_norm.astype(dtype), w.k_norm.astype(dtype), cos, sin, cfg)
    attn = attention(q, k, _heads(v, cfg.heads, cfg.head_dim)).reshape(x.shape[0], x.shape[1], H)
    act = swiglu(gate, up)
    cat = np.concatenate([attn, act], axis=-1)
    return x + mod["single_gate"] * _project(cat, w.out, e4m3 == "all", dtype, stored_bf16=True)


def final_layer(x_img, shift, scale, w_proj, cfg: Config, dtype=np.float64) -> np.ndarray:
    """Reading R16: (1 + scale) LN(x) + shift, then Linear(H -> in_channels)."""
    y = adaln(x_img.astype(dtype), shift, scale, cfg.eps)
    return y @ w_proj.astype(dtype).T


# ----------------------------------------------------------------------------------
# e4m3 quantisation (reading R26 of the [pyref] KleinTT constructor's precision knob).
# The pages name the knob without a format; the format here is the common 8-bit float
# with 1 sign bit, 4 exponent bits (bias 7) and 3 mantissa bits: normal values
# (-1)^s 2^(e-7) (1 + m/8) for e in 1..15 (e = 15, m = 7 is NaN, so the largest finite
# value is 1.75 * 2^8 = 448), subnormals (-1)^s 2^-6 (m/8) for e = 0.
# ----------------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_decode(code: int) -> float:
    """The value of one e4m3 byte (NaN for the two NaN codes)."""
    code = int(code)  # a numpy uint8 would wrap in e - 7 below
    s, e, m = (code >> 7) & 1, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return float("nan")
    mag = 2.0 ** -6 * (m / 8.0) if e == 0 else 2.0 ** (e - 7) * (1.0 + m / 8.0)
    return -mag if s else mag


def e4m3_encode(x: float) -> int:
    """Round x to the nearest e4m3 value, ties to even mantissa, saturating to +-448
    (finite inputs only).  Pure-Python: the grid is walked per binade."""
    sign = 0x80 if (x < 0 or (x == 0 and np.signbit(x))) else 0
    a = abs(float(x))
    if a >= E4M3_MAX:
        return sign | 0x7E
    if a < 2.0 ** -6:  # subnormal binade (and zero): steps of 2^-9
        q = _round_half_even(a / 2.0 ** -9)
        return sign | q  # q == 8 is the smallest normal, code 0x08, by construction
    e = int(np.floor(np.log2(a)))
    while 2.0 ** e > a:  # guard the log2 rounding at binade edges
        e -= 1
    while 2.0 ** (e + 1) <= a:
        e += 1
    q = _round_half_even(a / 2.0 ** (e - 3))  # 8 .. 16
    if q == 16:
        e, q = e + 1, 8
    code = ((e + 7) << 3) | (q - 8)
    return sign | min(code, 0x7E)


def _round_half_even(t: float) -> int:
    f = int(np.floor(t))
    r = t - f
    if r > 0.5 or (r == 0.5 and f % 2 == 1):
        f += 1
    return f


def _row_scales(x: np.ndarray):
    """scale = max|row| / 448 (1 for an all-zero row) and its reciprocal, both computed in
    fp32 as the quantiser does (reading R26)."""
    amax = np.abs(x).max(axis=-1).astype(np.float32)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    inv = (np.float32(1.0) / scale).astype(np.float32)
    return scale, inv


def quantize_rows_e4m3(w: np.ndarray):
    """Per-row e4m3 quantisation as the library's weight preparation defines it, in fp32
    arithmetic: scale = max|w[r,:]| / 448 (1 for an all-zero row), q = e4m3(w * (1/scale)).
    Returns (codes uint8 [rows, cols], scale float32 [rows])."""
    w = np.asarray(w, dtype=np.float32)
    scale, inv = _row_scales(w)
    scaled = (w * inv[:, None]).astype(np.float32)
    codes = np.array([[e4m3_encode(v) for v in row] for row in scaled], dtype=np.uint8)
    return codes, scale


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """The nearest e4m3 value of every element of a float32 array (ties to even,
    saturating to +-448), as float32 (every e4m3 value is exact in float32): the same map
    as e4m3_decode(e4m3_encode(.)), for whole arrays.  Magnitudes are first clipped to 448,
    the largest finite value.  From 2^-6 up, e4m3 keeps 3 significand bits, so the float32
    value is rounded to the top 3 of its 23 stored significand bits: add half of the 20
    dropped bits' weight (0x80000, one less when the lowest kept bit is even) and clear
    them; a carry out of the significand moves to the next binade, as it should.  Below
    2^-6 the grid is the subnormal step 2^-9: x * 2^9 rounded to an integer (exact
    scaling, rint is ties-to-even)."""
    x = np.asarray(x, dtype=np.float32)
    a = np.minimum(np.abs(x), np.float32(E4M3_MAX))
    u = a.view(np.uint32)
    t = np.right_shift(u, np.uint32(20))
    np.bitwise_and(t, np.uint32(1), out=t)
    t += np.uint32(0x7FFFF)
    t += u
    np.bitwise_and(t, np.uint32(0xFFF00000), out=t)
    q = t.view(np.float32)
    small = a < np.float32(2.0 ** -6)
    if small.any():
        q[small] = np.rint(a[small] * np.float32(512.0)) * np.float32(1.0 / 512.0)
    return np.copysign(q, x, out=q)


def quantize_rows_e4m3_values(x: np.ndarray):
    """Per-row e4m3 quantisation of the last axis in the kernel's precision (fp32: the
    scale, its reciprocal and x * (1/scale) are fp32 values, reading R26).  Returns the
    decoded e4m3 values (float32, exact; same shape as x) and the scales (float32, x.shape[:-1]):
    x ~ values * scale[..., None].  The same arithmetic as quantize_rows_e4m3, for whole
    arrays."""
    x = np.asarray(x, dtype=np.float32)
    scale, inv = _row_scales(x)
    return e4m3_round((x * inv[..., None]).astype(np.float32)), scale


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 value, ties to even (finite inputs), returned as
    float32: bf16 keeps the top 16 bits of the fp32 pattern, so the rounding adds half of
    the dropped 16-bit field (0x8000, one less when the kept part is even) and truncates.
    The storage rounding of the GPU path's inter-kernel tensors (reading R18); the oracle
    applies it only where a stored value feeds a quantiser, so that both sides take the
    quantiser's decisions on the same input (reading R26)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(f.shape)


def linear_e4m3(a: np.ndarray, w: np.ndarray, dtype=np.float64) -> np.ndarray:
    """a @ w^T with both operands in e4m3 (reading R26): a quantised per token row (its
    last axis), w [out, in] per output row, the products of the decoded values summed in
    `dtype`, then dequantised: y[m, n] = (sum_k qa[m, k] qw[n, k]) sa[m] sw[n]."""
    qa, sa = quantize_rows_e4m3_values(a)
    qw, sw = quantize_rows_e4m3_values(w)
    y = qa.astype(dtype) @ qw.astype(dtype).T
    return y * sa[..., None].astype(dtype) * sw.astype(dtype)


# ----------------------------------------------------------------------------------
# The whole step and the 4-step loop
# ----------------------------------------------------------------------------------
@dataclass
class Weights:
    cfg: Config
    t_in: np.ndarray          # [H, 256]
    t_out: np.ndarray         # [H, H]
    mod: np.ndarray           # [17H, H]
    x_emb: np.ndarray         # [H, in_channels]
    ctx_emb: np.ndarray       # [H, txt_dim]
    proj_out: np.ndarray      # [in_channels, H]
    dual: list = field(default_factory=list)     # [(StreamWeights img, StreamWeights txt)]
    single: list = field(default_factory=list)   # [SingleWeights]


def dit_step(w: Weights, img_tokens, ref_tokens, txt_emb, sigma, ids, dtype=np.float64,
             n_dual=None, n_single=None, e4m3=None) -> np.ndarray:
    """One velocity evaluation ([card] task table: one DiT call per step, no CFG).

    img_tokens [B, n_img, C], ref_tokens [B, n_ref, C] or None, txt_emb [B, n_txt, 7680],
    sigma [B], ids [N, 4].  Returns the velocity of the target-image rows [B, n_img, C].
    e4m3 ("fused" / "all") runs the blocks' projections in e4m3 (reading R26); the
    embedders, the modulation and the final projection stay unquantised.
    The joint sequence is [txt | img | ref] (reading R1); reference tokens are clean
    latents, embedded by the same image embedder (reading R22).
    """
    cfg = w.cfg
    cast = lambda a: np.asarray(a).astype(dtype)
    n_txt, n_img = txt_emb.shape[1], img_tokens.shape[1]
    parts = [cast(txt_emb) @ cast(w.ctx_emb).T, cast(img_tokens) @ cast(w.x_emb).T]
    if ref_tokens is not None and ref_tokens.shape[1] > 0:
        parts.append(cast(ref_tokens) @ cast(w.x_emb).T)
    x = np.concatenate(parts, axis=1)
    m = modulation(sigma, w.t_in, w.t_out, w.mod, cfg, dtype)
    mod = split_modulation(m, cfg.hidden)
    cos, sin = rope_table(ids, cfg.axes_dim, cfg.rope_theta)
    cos, sin = cos.astype(dtype), sin.astype(dtype)
    nd = len(w.dual) if n_dual is None else n_dual
    ns = len(w.single) if n_single is None else n_single
    for i in range(nd):
        x = dual_block(x, n_txt, w.dual[i][0], w.dual[i][1], mod, cos, sin, cfg, dtype,
                       e4m3="all" if e4m3 == "all" else None)
    for i in range(ns):
        x = single_block(x, w.single[i], mod, cos, sin, cfg, dtype, e4m3=e4m3)
    x_img = x[:, n_txt:n_txt + n_img]
    return final_layer(x_img, mod["final_shift"], mod["final_scale"], w.proj_out, cfg, dtype)


def sigma_schedule(sigma0: float, steps: int = 4) -> np.ndarray:
    """Reading R19: sigma_k = sigma0 (1 - k/steps), k = 0..steps, ending at 0.
    The pages name compute_empirical_mu ([pyref] Modules: host.py) without its formula,
    so no time shift is applied.  Parity unpinned against upstream (no formula)."""
    k = np.arange(steps + 1, dtype=np.float64)
    return sigma0 * (1.0 - k / steps)


def euler_update(x, v, sigma_cur, sigma_next):
    """Flow-matching Euler step x <- x + (sigma_next - sigma_cur) v."""
    return x + (sigma_next - sigma_cur) * v


def denoise(w: Weights, x0, ref_tokens, txt_emb, ids, sigmas, dtype=np.float64, e4m3=None):
    """The 4-step loop ([card]: steps fixed at 4, each step one DiT call).  e4m3 is passed to
    every step (reading R26 of the precision knob); the Euler update itself is unquantised."""
    x = np.asarray(x0).astype(dtype)
    B = x.shape[0]
    for k in range(len(sigmas) - 1):
        v = dit_step(w, x, ref_tokens, txt_emb, np.full(B, sigmas[k]), ids, dtype, e4m3=e4m3)
        x = euler_update(x, v, sigmas[k], sigmas[k + 1])
    return x

