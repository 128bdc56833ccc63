"""Test helpers: turn the seeded synthetic tensors into the oracle's numpy structures
and compare results.  Shared by CPU and GPU tests; holds no arithmetic of the method."""
from __future__ import annotations

import numpy as np
import torch

from oracle import dit_oracle as O


def to_np(t, dtype=np.float64):
    if t is None:
        return None
    return t.detach().to("cpu", torch.float32).numpy().astype(dtype)


def oracle_config(wd) -> O.Config:
    return O.Config(hidden=wd.hidden, heads=wd.heads, head_dim=wd.head_dim,
                    mlp_hidden=wd.mlp_hidden, n_dual=wd.n_dual, n_single=wd.n_single,
                    in_channels=wd.in_channels, txt_dim=wd.txt_dim)


def oracle_stream(w, dtype=np.float64) -> O.StreamWeights:
    return O.StreamWeights(**{k: to_np(v, dtype) for k, v in w.items()})


def oracle_single(w, dtype=np.float64) -> O.SingleWeights:
    return O.SingleWeights(**{k: to_np(v, dtype) for k, v in w.items()})


def oracle_weights(wd, w, dtype=np.float64) -> O.Weights:
    cfg = oracle_config(wd)
    return O.Weights(cfg=cfg, t_in=to_np(w["mod"]["t_in"], dtype), t_out=to_np(w["mod"]["t_out"], dtype),
                     mod=to_np(w["mod"]["mod"], dtype), x_emb=to_np(w["x_emb"], dtype),
                     ctx_emb=to_np(w["ctx_emb"], dtype), proj_out=to_np(w["proj_out"], dtype),
                     dual=[(oracle_stream(a, dtype), oracle_stream(b, dtype)) for a, b in w["dual"]],
                     single=[oracle_single(s, dtype) for s in w["single"]])


def cosine(a, b) -> float:
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


def read_kv(path):
    out = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        k, v = [s.strip() for s in line.split("=", 1)]
        out[k] = v
    return out


def read_rows(path):
    rows = []
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if line:
            rows.append([int(x) for x in line.split()])
    return np.asarray(rows, dtype=np.int64)


def read_step_golden(path):
    """Parse a step golden: `key = value` lines and `v <row> <token> <values...>` lines."""
    kv, vel = {}, {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        if line.startswith("v "):
            parts = line.split()
            vel[(int(parts[1]), int(parts[2]))] = np.asarray([float(x) for x in parts[3:]], np.float64)
        else:
            k, v = [s.strip() for s in line.split("=", 1)]
            kv[k] = v
    return kv, vel


def input_fingerprints(logical: dict, inp: dict) -> dict:
    """float64 (sum, sum of squares) of the seeded step inputs, per tensor group: lets a test
    tell a changed input stream from a changed result.  `logical` None: activations only."""
    def acc(tensors):
        s = q = 0.0
        for t in tensors:
            if t is None:
                continue
            d = t.double()
            s += float(d.sum())
            q += float((d * d).sum())
        return s, q
    groups = {
        "img_tokens": [inp["img_tokens"]],
        "ref_tokens": [inp["ref_tokens"]],
        "txt_emb": [inp["txt_emb"]],
    }
    if logical is not None:
        groups.update({
            "mod": list(logical["mod"].values()),
            "embedders": [logical["x_emb"], logical["ctx_emb"], logical["proj_out"]],
            "dual": [t for pair in logical["dual"] for sw in pair for t in sw.values()],
            "single": [t for sw in logical["single"] for t in sw.values()],
        })
    return {k: acc(v) for k, v in groups.items()}


def check_fingerprints(mine: dict, kv: dict):
    """Compare input fingerprints with a golden's `fingerprint.<group> = sum sumsq` lines.

    The bounds allow for float64 summation order only (about 1e-12 relative).  A different
    stream moves the sum by about sqrt(sumsq) and the sum of squares by about
    sqrt(2/n) relative; the last-place drift of a float32 sampler across hosts moved the sum
    of 4.2 M latent values by ~4e-5 sqrt(sumsq)."""
    for k, (s, q) in mine.items():
        ws, wq = (float(x) for x in kv[f"fingerprint.{k}"].split())
        assert abs(s - ws) <= 1e-6 * wq ** 0.5 and abs(q - wq) <= 1e-10 * wq, (k, s, ws, q, wq)


def block_metrics(got, want, xin) -> dict:
    """Parity figures of one block output against the oracle, all on [1, N, H] arrays.

    max_abs, cos: of the whole output x_out.  The output is dominated by the unchanged
    residual x_in, so the block's own update u = x_out - x_in is also compared: upd_cos
    over the whole update, and the largest rms error of the update over any one token row
    (row_err) and over any one output column (col_err), each relative to the rms of the
    whole update.  A wrong scale of one token row or of one output channel (a
    dequantisation on the wrong index) shows there in full, while it moves the
    whole-tensor figures by only its share of the rows or columns.  The oracle's output is
    rounded to bf16 first for the update figures, as the GPU's is."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    xin = np.asarray(xin, np.float64)
    want_q = torch.from_numpy(np.asarray(want, np.float32)).to(torch.bfloat16).double().numpy()
    du, wu = got - xin, want_q - xin
    err = (du - wu).reshape(-1, du.shape[-1])
    u_rms = max(float(np.sqrt((wu * wu).mean())), 1e-30)
    row = np.sqrt((err * err).mean(axis=1)) / u_rms
    col = np.sqrt((err * err).mean(axis=0)) / u_rms
    return {"max_abs": max_abs(got, want), "cos": cosine(got, want), "upd_cos": cosine(du, wu),
            "row_err": float(row.max()), "col_err": float(col.max())}


def block_metrics_fail(m: dict, bars: dict) -> list:
    """Names of the figures of `m` outside `bars` (max_abs, row_err, col_err: upper
    bounds; cos, upd_cos: lower bounds)."""
    bad = []
    for k, lim in bars.items():
        v = m[k]
        if (k in ("cos", "upd_cos") and not v >= lim) or (k not in ("cos", "upd_cos") and not v <= lim):
            bad.append(k)
    return bad


# ---- parity bars of a block output against the oracle (shared by the GPU tests and the
# CPU test that plants wrong scales in a copy of the oracle's e4m3 path)
#
# bf16 path against the unquantised oracle.  max_abs 3e-2, cos 0.999: the acceptance
# bars.  upd_cos 0.99: the update u = x_out - x_in differs from the oracle's by the
# GPU's bf16 storage of Q/K/V, P, the attention output, the activations (relative
# rounding <= 2^-9 each) and by the bf16 output itself, whose one-ulp disagreements
# (ulp 2^-8 at |x| ~ 1) weigh most where the update is smallest, the hidden-256 blocks
# (update rms ~ 10 ulps): a relative rms error of ~5 % there, cosine ~0.9988; 0.99
# allows 14 %.  At klein width (hidden >= 3072, updates ~5x larger against the same
# ulp) the error of any one token row or output column, relative to the update's rms,
# is ~1 % (bf16 intermediates) and ~2 % (columns, the maximum over 3072): bars 0.05.
BF16_BARS = {"max_abs": 3e-2, "cos": 0.999, "upd_cos": 0.99}
BF16_ROWCOL_BARS = {"row_err": 0.05, "col_err": 0.05}
# e4m3 path against the e4m3-aware oracle (reading R26: same quantiser, same scales, same
# decisions in fp32 on the values the GPU feeds it).  What is left is the bf16 path's
# error plus the quantiser decisions that differ because the two sides' inputs differ
# by that error: a decision flips where an input lies within the bf16 path's ~1 %
# discrepancy of a rounding midpoint of the e4m3 grid (step 2^-3 of the binade), for a
# few % of the elements of a twice-quantised dual-block chain, and each flip moves one
# element by one e4m3 step.  Relative to the update's rms that is ~0.03 per row and up
# to ~0.07 for the worst of 3072-4096 columns: bars 0.12 (a wrong scale by 25 % on one
# token row, or on one output column of median size, gives 0.16-0.25; see
# test_e4m3_bars_reject_a_wrong_scale).  One flip at a row's largest activation (step
# 1/14 of the row maximum, act maxima ~20, |w| <= 0.09, |gate| <= 0.35) moves an output by
# ~0.05: max_abs 0.15 allows three.  cos and upd_cos as for bf16.
E4M3_BARS = {"max_abs": 0.15, "cos": 0.999, "upd_cos": 0.99}
E4M3_ROWCOL_BARS = {"row_err": 0.12, "col_err": 0.12}
# The accuracy report of the e4m3 path against the unquantised oracle: e4m3 rounds each
# operand by up to 2^-4 relative (rms ~2.6 %), so each projection carries ~4 % rms and a
# block's update ~7 % (cosine ~0.9975 measured); 0.97 allows 24 %.  max_abs 0.25: the
# quantisation of the row maxima as above, unaligned between the two sides.
E4M3_ACCURACY_BARS = {"max_abs": 0.25, "cos": 0.999, "upd_cos": 0.97}
