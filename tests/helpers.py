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
    over the whole update, and the worst relative rms error of the update over any one
    token row (row_rel) and over any one output column (col_rel).  A wrong scale of one
    token row or one output channel (a dequantisation on the wrong index) shows there in
    full, while it moves the whole-tensor figures by only its share of the rows or columns.
    The oracle's output is rounded to bf16 first for the update figures, as the GPU's is."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    xin = np.asarray(xin, np.float64)
    want_q = torch.from_numpy(np.asarray(want, np.float32)).to(torch.bfloat16).double().numpy()
    du, wu = got - xin, want_q - xin
    err = du - wu
    rms = lambda a, ax: np.sqrt((a * a).mean(axis=ax))
    row = rms(err, -1) / np.maximum(rms(wu, -1), 1e-30)
    col = rms(err.reshape(-1, err.shape[-1]), 0) / np.maximum(rms(wu.reshape(-1, wu.shape[-1]), 0), 1e-30)
    return {"max_abs": max_abs(got, want), "cos": cosine(got, want), "upd_cos": cosine(du, wu),
            "row_rel": float(row.max()), "col_rel": float(col.max())}


def block_metrics_fail(m: dict, bars: dict) -> list:
    """Names of the figures of `m` outside `bars` (max_abs, row_rel, col_rel: upper
    bounds; cos, upd_cos: lower bounds)."""
    bad = []
    for k, lim in bars.items():
        v = m[k]
        if (k in ("cos", "upd_cos") and not v >= lim) or (k not in ("cos", "upd_cos") and not v <= lim):
            bad.append(k)
    return bad
