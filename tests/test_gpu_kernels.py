"""GPU parity of each kernel against the oracle, through the C ABI, on seeded inputs at
sizes the oracle finishes in seconds that span several tiles and a ragged tail.

Tolerances: every output is stored as bf16 (relative rounding 2^-9), inputs are the same
bf16 values on both sides and all accumulation is fp32 on the GPU, so the bound is a
few bf16 ulps of the output's magnitude: max-abs <= 3e-2 and cosine >= 0.9999 (0.999 for
attention, whose P is rounded to bf16 before the PV product).
"""
import numpy as np
import pytest
import torch

from oracle import dit_oracle as O
from diffusion_transformer_step_gb300 import synth
import helpers as Hx

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def dit():
    from diffusion_transformer_step_gb300 import build_lib
    build_lib.build()
    from diffusion_transformer_step_gb300 import dit as d
    d.lib()
    return d


@pytest.fixture()
def ws():
    t = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    return t


def _check_status(dit, ws):
    st, where = dit.dit_sync_status(ws)
    assert st == dit.DIT_OK, f"device wait gave up at site {where:#x}"


def _randn(shape, std=1.0, seed=0, mean=0.0):
    g = synth.generator(seed)
    return synth.normal(shape, std, g, mean=mean)


def _cmp(got, want, atol=3e-2, cos_min=0.9999):
    got = Hx.to_np(got)
    err = Hx.max_abs(got, want)
    cs = Hx.cosine(got, want)
    assert np.isfinite(got).all()
    assert err <= atol and cs >= cos_min, (err, cs)
    return err, cs


@pytest.mark.parametrize("n_txt,grid,refs", [(32, (8, 8), ()), (512, (64, 64), ()), (512, (68, 120), ((64, 64),))])
def test_rope_table(dit, n_txt, grid, refs):
    nref = sum(a * b for a, b in refs)
    shape = dit.make_shape(1, n_txt, grid[0] * grid[1], nref)
    ids = dit.dit_token_ids(shape, grid[0], grid[1], refs)
    N = ids.shape[0]
    table = torch.empty((N, 64, 2), dtype=torch.float32, device=DEV)
    dit.dit_rope_table(dit.dit_config_klein(), ids.to(DEV), N, table)
    torch.cuda.synchronize()
    c, s = O.rope_table(O.token_ids(n_txt, grid[0], grid[1], refs))
    t = table.cpu().numpy().astype(np.float64)
    # fp64 angle rounded once to fp32
    np.testing.assert_allclose(t[..., 0], c, rtol=0, atol=1.2e-7)
    np.testing.assert_allclose(t[..., 1], s, rtol=0, atol=1.2e-7)


@pytest.mark.parametrize("hidden,rows,split,batch", [(256, 96, 32, 1), (3072, 300, 77, 2), (3072, 4608, 512, 1)])
def test_adaln(dit, hidden, rows, split, batch):
    x_rows = rows + 5
    x = _randn((batch, x_rows, hidden), 1.5, seed=1, mean=0.3).to(DEV)
    mod = _randn((batch, 4, hidden), 0.1, seed=2).to(DEV)
    y = torch.empty((batch, rows, hidden), dtype=torch.bfloat16, device=DEV)
    dit.dit_adaln(batch, rows, hidden, x, x_rows, 3, split, mod[:, 0], mod[:, 1], mod[:, 2], mod[:, 3],
                  4 * hidden, 1e-6, y)
    torch.cuda.synchronize()
    xn, mn = Hx.to_np(x), Hx.to_np(mod)
    want = np.empty((batch, rows, hidden))
    for b in range(batch):
        xs = xn[b, 3:3 + rows]
        want[b, :split] = O.adaln(xs[:split], mn[b, 0], mn[b, 1], 1e-6)
        want[b, split:] = O.adaln(xs[split:], mn[b, 2], mn[b, 3], 1e-6)
    _cmp(y, want)


@pytest.mark.parametrize("axes,theta", [((16, 56, 56, 0), 10000.0), ((0, 64, 32, 32), 2000.0)])
def test_rope_table_other_axis_splits(dit, axes, theta):
    """The table for other splits of the 128 head dims over the four axes (one of them empty)
    and another theta: every pair's cos / sin against the oracle's table of that split."""
    n_txt, grid, refs = 16, (6, 10), ((3, 4),)
    shape = dit.make_shape(1, n_txt, grid[0] * grid[1], 12)
    ids = dit.dit_token_ids(shape, grid[0], grid[1], refs)
    N = ids.shape[0]
    cfg = dit.dit_config_klein()
    for i, d in enumerate(axes):
        cfg.axes_dim[i] = d
    cfg.rope_theta = theta
    table = torch.empty((N, 64, 2), dtype=torch.float32, device=DEV)
    dit.dit_rope_table(cfg, ids.to(DEV), N, table)
    torch.cuda.synchronize()
    c, s = O.rope_table(O.token_ids(n_txt, grid[0], grid[1], refs), axes, theta)
    t = table.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(t[..., 0], c, rtol=0, atol=1.2e-7)
    np.testing.assert_allclose(t[..., 1], s, rtol=0, atol=1.2e-7)


@pytest.mark.parametrize("hidden", [256 * v for v in (1, 2, 3, 4, 5, 6, 8, 10, 12, 14, 16)])
def test_adaln_every_supported_width(dit, hidden):
    """Every hidden width the kernel is instantiated for (hidden / 256 vectors of 8 per lane),
    two batch rows, a ragged row count and a split, every element against the oracle."""
    batch, rows, split = 2, 37, 11
    x = _randn((batch, rows, hidden), 1.5, seed=61, mean=-0.4).to(DEV)
    mod = _randn((batch, 4, hidden), 0.1, seed=62).to(DEV)
    y = torch.empty((batch, rows, hidden), dtype=torch.bfloat16, device=DEV)
    dit.dit_adaln(batch, rows, hidden, x, rows, 0, split, mod[:, 0], mod[:, 1], mod[:, 2], mod[:, 3], 4 * hidden,
                  1e-6, y)
    torch.cuda.synchronize()
    xn, mn = Hx.to_np(x), Hx.to_np(mod)
    want = np.empty((batch, rows, hidden))
    for b in range(batch):
        want[b, :split] = O.adaln(xn[b, :split], mn[b, 0], mn[b, 1], 1e-6)
        want[b, split:] = O.adaln(xn[b, split:], mn[b, 2], mn[b, 3], 1e-6)
    _cmp(y, want)


def test_adaln_at_the_row_limit(dit):
    """adaLN at the library's token limit (2^20 rows less a ragged 13) for two batch rows,
    hidden 256, with the split between the two modulation pairs in the middle: ~2 x 2^20
    rows streamed through each CTA's ring.  Sampled rows on both sides of the split, at
    the start and the end, against the oracle."""
    batch, rows, hidden = 2, (1 << 20) - 13, 256
    split = rows // 2 + 7
    x = _randn((batch, rows, hidden), 1.5, seed=51, mean=0.3)
    mod = _randn((batch, 4, hidden), 0.1, seed=52)
    y = torch.empty((batch, rows, hidden), dtype=torch.bfloat16, device=DEV)
    md = mod.to(DEV)
    dit.dit_adaln(batch, rows, hidden, x.to(DEV), rows, 0, split, md[:, 0], md[:, 1], md[:, 2], md[:, 3],
                  4 * hidden, 1e-6, y)
    torch.cuda.synchronize()
    sel = [0, 1, 31, 32, split - 1, split, split + 1, rows - 300, rows - 13, rows - 1]
    xn, mn = Hx.to_np(x[:, sel]), Hx.to_np(mod)
    want = np.empty((batch, len(sel), hidden))
    for b in range(batch):
        for i, r in enumerate(sel):
            lo = r < split
            want[b, i] = O.adaln(xn[b, i:i + 1], mn[b, 0 if lo else 2], mn[b, 1 if lo else 3], 1e-6)[0]
    _cmp(y[:, sel], want)


WIDE_MOD = synth.Widths(hidden=4096, heads=32, head_dim=128, mlp_hidden=12288, n_dual=1, n_single=1)


# hidden 768 and 1536: eight batch rows of a 1536-wide input fill exactly the default 48 KB
# of dynamic shared memory of the GEMV
MOD_768 = synth.Widths(hidden=768, heads=6, head_dim=128, mlp_hidden=2304, n_dual=1, n_single=1)
MOD_1536 = synth.Widths(hidden=1536, heads=12, head_dim=128, mlp_hidden=4608, n_dual=1, n_single=1)


@pytest.mark.parametrize("wd,batch", [(synth.TINY, 1), (synth.TINY, 3), (synth.KLEIN, 1), (synth.KLEIN, 3),
                                      (synth.KLEIN, 11), (WIDE_MOD, 8), (MOD_768, 8), (MOD_1536, 8),
                                      (MOD_1536, 5)],
                         ids=lambda v: getattr(v, "hidden", v))
def test_modulation(dit, wd, batch, ws):
    """Every element of the modulation vector against the oracle; batch 11 runs as launches
    of 8 and 3 rows, batch 8 at hidden 4096 fills one launch's largest instantiation."""
    g = synth.generator(7)
    mw = synth.mod_weights(wd, g)
    w = dit.dit_weights()
    w.cfg = dit.make_config(hidden=wd.hidden, heads=wd.heads, mlp_hidden=wd.mlp_hidden)
    dev = {k: v.to(DEV) for k, v in mw.items()}
    w.mod.t_in, w.mod.t_out, w.mod.mod = dev["t_in"].data_ptr(), dev["t_out"].data_ptr(), dev["mod"].data_ptr()
    sigma = torch.tensor([0.93, 0.51, 0.0, 1.0, 0.25, 0.7, 0.33, 0.05, 0.88, 0.6, 0.12][:batch], dtype=torch.float32)
    out = torch.empty((batch, 17 * wd.hidden), dtype=torch.bfloat16, device=DEV)
    dit.dit_modulation(w, sigma.to(DEV), batch, out, ws, ws.numel())
    _check_status(dit, ws)
    want = O.modulation(sigma.numpy().astype(np.float64), Hx.to_np(mw["t_in"]), Hx.to_np(mw["t_out"]),
                        Hx.to_np(mw["mod"]), O.Config(hidden=wd.hidden))
    _cmp(out, want, atol=1e-2)


@pytest.mark.parametrize("batch,rows,n,k", [(1, 128, 256, 64), (2, 300, 288, 320), (1, 1000, 768, 3072),
                                            (3, 17, 128, 7680), (1, 70, 32, 8), (2, 130, 64, 40)])
def test_linear_store(dit, batch, rows, n, k, ws):
    a = _randn((batch, rows, k), 1.0, seed=3).to(DEV)
    w = _randn((n, k), 0.05, seed=4).to(DEV)
    ld = n + 32
    out = torch.full((batch, rows, ld), 7.0, dtype=torch.bfloat16, device=DEV)
    dit.dit_linear(batch, rows, n, k, a, w, out, ld, dit.DIT_EPI_STORE, None, 0, ws, ws.numel())
    _check_status(dit, ws)
    want = Hx.to_np(a) @ Hx.to_np(w).T
    scale = np.abs(want).max()
    _cmp(out[..., :n], want, atol=1e-2 * scale)
    assert (out[..., n:] == 7.0).all()  # columns past n_out untouched


def test_linear_at_the_row_limit(dit, ws):
    """The GEMM at the library's token limit (2^20 rows less a ragged 13), two batches, a
    ragged n (96) and k (72): 16384 row tiles.  Sampled rows of both batches (first tiles,
    the middle, the last full tile, the ragged tail) against the product in fp64."""
    batch, rows, n, k = 2, (1 << 20) - 13, 96, 72
    a = _randn((batch, rows, k), 1.0, seed=41)
    w = _randn((n, k), 0.05, seed=42)
    out = torch.zeros((batch, rows, n), dtype=torch.bfloat16, device=DEV)
    dit.dit_linear(batch, rows, n, k, a.to(DEV), w.to(DEV), out, n, dit.DIT_EPI_STORE, None, 0, ws, ws.numel())
    _check_status(dit, ws)
    sel = [0, 1, 127, 128, 255, 256, rows // 2, rows // 2 + 129, rows - 300, rows - 129, rows - 13, rows - 1]
    want = Hx.to_np(a[:, sel]) @ Hx.to_np(w).T
    _cmp(out[:, sel], want, atol=1e-2 * np.abs(want).max())


@pytest.mark.parametrize("batch,rows,n,k", [(1, 256, 256, 256), (2, 300, 3072, 320)])
def test_linear_gated_residual(dit, batch, rows, n, k, ws):
    a = _randn((batch, rows, k), 1.0, seed=5).to(DEV)
    w = _randn((n, k), 0.05, seed=6).to(DEV)
    x0 = _randn((batch, rows, n), 1.0, seed=7)
    gate = _randn((batch, 3 * n), 0.1, seed=8)
    x = x0.clone().to(DEV)
    gd = gate.to(DEV)
    dit.dit_linear(batch, rows, n, k, a, w, x, n, dit.DIT_EPI_GATED_RESIDUAL, gd[:, n:], 3 * n, ws, ws.numel())
    _check_status(dit, ws)
    want = Hx.to_np(x0) + Hx.to_np(gate)[:, None, n:2 * n] * (Hx.to_np(a) @ Hx.to_np(w).T)
    _cmp(x, want)


@pytest.mark.parametrize("batch,rows,f,k", [(1, 128, 128, 64), (2, 300, 768, 256), (1, 520, 9216, 3072)])
def test_linear_swiglu_packed(dit, batch, rows, f, k, ws):
    a = _randn((batch, rows, k), 1.0, seed=9).to(DEV)
    w = _randn((2 * f, k), 0.05, seed=10)
    wp = torch.empty((2 * f, k), dtype=torch.bfloat16, device=DEV)
    dit.dit_pack_mlp_in(w.to(DEV), wp, f, k)
    out = torch.zeros((batch, rows, f), dtype=torch.bfloat16, device=DEV)
    dit.dit_linear(batch, rows, f, k, a, wp, out, f, dit.DIT_EPI_SWIGLU, None, 0, ws, ws.numel())
    _check_status(dit, ws)
    h = Hx.to_np(a) @ Hx.to_np(w).T
    want = O.swiglu(h[..., :f], h[..., f:])
    _cmp(out, want, atol=1e-2 * max(1.0, np.abs(want).max()))


@pytest.mark.parametrize("batch,heads,n,qscale", [(1, 1, 128, 1.0), (1, 2, 300, 1.0), (2, 3, 1000, 1.0),
                                                  (1, 2, 700, 6.0), (1, 1, 5, 1.0)])
def test_attention(dit, batch, heads, n, qscale, ws):
    q = _randn((batch, heads, n, 128), qscale, seed=11)
    k = _randn((batch, heads, n, 128), 1.0, seed=12)
    v = _randn((batch, heads, n, 128), 1.0, seed=13)
    ld = heads * 128 + 64
    out = torch.zeros((batch, n, ld), dtype=torch.bfloat16, device=DEV)
    dit.dit_attention(batch, heads, n, q.to(DEV), k.to(DEV), v.to(DEV), out, ld, ws, ws.numel())
    _check_status(dit, ws)
    t = lambda z: Hx.to_np(z).transpose(0, 2, 1, 3)  # [B, N, heads, D]
    want = O.attention(t(q), t(k), t(v)).reshape(batch, n, heads * 128)
    _cmp(out[..., :heads * 128], want, atol=3e-2, cos_min=0.999)
    assert (out[..., heads * 128:] == 0).all()


def test_attention_at_the_sequence_limit(dit, ws):
    """Attention at the library's token limit (2^20 tokens less a ragged 13): 8192 key
    blocks through the two-slot ring and 4096 CTAs.  Sampled query rows (first tiles, the
    middle, the last full tile and the ragged tail) against the oracle over every key, in
    fp32 for this size."""
    n = (1 << 20) - 13
    q = _randn((1, 1, n, 128), 1.0, seed=31)
    k = _randn((1, 1, n, 128), 1.0, seed=32)
    v = _randn((1, 1, n, 128), 1.0, seed=33)
    out = torch.zeros((1, n, 128), dtype=torch.bfloat16, device=DEV)
    dit.dit_attention(1, 1, n, q.to(DEV), k.to(DEV), v.to(DEV), out, 128, ws, ws.numel())
    _check_status(dit, ws)
    rows = [0, 1, 127, 128, 255, 256, n // 2, n // 2 + 129, n - 300, n - 141, n - 129, n - 13, n - 1]
    qs = Hx.to_np(q[0, 0, rows], np.float32)[None, :, None, :]
    kk = Hx.to_np(k[0, 0], np.float32)[None, :, None, :]
    vv = Hx.to_np(v[0, 0], np.float32)[None, :, None, :]
    want = O.attention(qs, kk, vv)[0, :, 0, :]
    _cmp(out[0, rows], want, atol=3e-2, cos_min=0.999)


def test_bounded_wait_reports_timeout_and_context_survives(dit, ws):
    """A device wait that can never complete gives up after its limit: the status word
    reports DIT_ERR_TIMEOUT with the waiting site, and later work on the GPU still runs."""
    import time
    t0 = time.perf_counter()
    dit.dit_selftest_wait_timeout(ws, ws.numel(), 20000)
    st, where = dit.dit_sync_status(ws)
    assert st == dit.DIT_ERR_TIMEOUT and where == 0x901
    assert time.perf_counter() - t0 < 5.0
    st, _ = dit.dit_sync_status(ws)          # cleared by the previous read
    assert st == dit.DIT_OK
    test_attention(dit, 1, 1, 128, 1.0, ws)   # the context is still usable


def test_quantize_rows_fp8_bit_exact(dit):
    """dit_quantize_rows_fp8 against the oracle's e4m3 quantiser, byte for byte: fp32
    scale = max|row| / 448, fp32 reciprocal and product, round-to-nearest-even with
    saturation.  Rows span small, large and all-zero values; 272 columns are not a multiple
    of the kernel's 256-thread stride."""
    rows, cols = 37, 272
    w = _randn((rows, cols), 0.05, seed=21)
    w[3] = 0.0
    w[5] *= 1.0e4
    w[9] *= 1.0e-6
    w[11, 7] = 3.0e4
    wd = w.to(DEV)
    q = torch.empty((rows, cols), dtype=torch.uint8, device=DEV)
    sc = torch.empty((rows,), dtype=torch.float32, device=DEV)
    dit.dit_quantize_rows_fp8(wd, rows, cols, q, sc)
    torch.cuda.synchronize()
    codes, scale = O.quantize_rows_e4m3(Hx.to_np(w, np.float32))
    assert np.array_equal(sc.cpu().numpy(), scale)
    got = q.cpu().numpy()
    bad = np.argwhere(got != codes)
    assert bad.size == 0, (bad[:5], got[tuple(bad[0])] if bad.size else None)
