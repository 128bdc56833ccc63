"""The C ABI without a GPU: the library loads, exports every symbol include/dit.h declares,
validates arguments before touching any device, and its host maths (token ids) equals
the oracle's bit for bit."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from oracle import dit_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dit.h")


@pytest.fixture(scope="module")
def dit():
    from diffusion_transformer_step_gb300 import build_lib
    build_lib.build()
    from diffusion_transformer_step_gb300 import dit as d
    d.lib()
    return d


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ ]*\*?\s+\**(dit_[a-z0-9_]+)\s*\(", src, re.M)))


def test_every_declared_symbol_is_exported(dit):
    names = declared_functions()
    assert len(names) >= 19, names
    L = dit.lib()
    for n in names:
        assert hasattr(L, n), n
    # and the binding wraps every one of them under the same name
    for n in names:
        assert n in dit._SIGS, n


def test_status_strings_and_klein_config(dit):
    for s in range(6):
        assert dit.dit_status_string(s)
    c = dit.dit_config_klein()
    assert (c.hidden, c.heads, c.head_dim, c.mlp_hidden, c.n_dual, c.n_single, c.in_channels, c.txt_dim) == \
        (3072, 24, 128, 9216, 5, 20, 128, 7680)
    assert abs(c.rope_theta - 2000.0) < 1e-3 and list(c.axes_dim) == [32, 32, 32, 32]


def test_token_ids_equal_oracle(dit):
    for n_txt, gh, gw, refs in ((512, 64, 64, ()), (512, 68, 120, ((64, 64),)), (3, 2, 3, ((1, 2), (2, 1))),
                                (7, 5, 3, ((2, 2), (3, 1), (1, 4)))):
        nref = sum(a * b for a, b in refs)
        shape = dit.make_shape(1, n_txt, gh * gw, nref)
        got = dit.dit_token_ids(shape, gh, gw, refs).numpy()
        np.testing.assert_array_equal(got, O.token_ids(n_txt, gh, gw, refs))


def test_token_ids_rejects_inconsistent_grid(dit):
    shape = dit.make_shape(1, 4, 10, 0)
    with pytest.raises(dit.DitError) as e:
        dit.dit_token_ids(shape, 3, 3)
    assert e.value.status == dit.DIT_ERR_INVALID_ARG
    # reference grids whose token counts overflow any sum, or exceed n_ref on the way
    shape = dit.make_shape(1, 4, 9, 6)
    for refs in (((2, 3), (1 << 30, 1 << 30)), ((1 << 30, 1 << 30), (1 << 30, 1 << 30)), ((4, 4),)):
        with pytest.raises(dit.DitError) as e:
            dit.dit_token_ids(shape, 3, 3, refs)
        assert e.value.status == dit.DIT_ERR_INVALID_ARG


def test_workspace_size_grows_with_shape(dit):
    c = dit.dit_config_klein()
    a = dit.dit_workspace_size(c, dit.make_shape(1, 512, 4096, 0))
    b = dit.dit_workspace_size(c, dit.make_shape(4, 512, 8160, 4096))
    assert 0 < a < b
    # 5 activation buffers of [N, H] + concat [N, H+F] dominate
    N, H, F = 4608, 3072, 9216
    assert a > N * H * 2 * 5 + N * (H + F) * 2


def test_workspace_size_at_the_largest_accepted_shape_does_not_wrap(dit):
    """Batch 64 and 2^20 tokens (the limits check_shape accepts) need ~10^14 bytes: the size
    must come out as that (64-bit arithmetic), and one row or token more is rejected."""
    c = dit.dit_config_klein()
    n_txt, n_img = 512, (1 << 20) - 512
    big = dit.dit_workspace_size(c, dit.make_shape(64, n_txt, n_img, 0))
    B, N, H, F = 64, 1 << 20, 3072, 9216
    assert big > B * N * (H + F) * 2 + B * N * H * 2 * 5
    assert big < 1 << 50
    assert big > dit.dit_workspace_size(c, dit.make_shape(63, n_txt, n_img, 0))
    for shape, want in ((dit.make_shape(65, n_txt, n_img, 0), dit.DIT_ERR_INVALID_ARG),
                        (dit.make_shape(1, n_txt, n_img + 1, 0), dit.DIT_ERR_UNSUPPORTED)):
        n = C.c_size_t(0)
        assert dit.lib().dit_workspace_size(C.byref(c), C.byref(shape), C.byref(n)) == want


def test_unsupported_configs_rejected(dit):
    shape = dit.make_shape(1, 8, 16, 0)
    big = (1 << 20) + 128  # past the GEMM width limit
    for field, val in (("head_dim", 64), ("hidden", 3000), ("mlp_hidden", 100), ("in_channels", 20),
                       ("txt_dim", 7), ("heads", 1 << 25), ("heads", 23), ("mlp_hidden", big),
                       ("in_channels", big), ("txt_dim", big)):
        c = dit.dit_config_klein()
        setattr(c, field, val)
        n = C.c_size_t(0)
        st = dit.lib().dit_workspace_size(C.byref(c), C.byref(shape), C.byref(n))
        assert st == dit.DIT_ERR_UNSUPPORTED, (field, st)
    c = dit.dit_config_klein()
    c.axes_dim[0] = 30
    assert dit.lib().dit_workspace_size(C.byref(c), C.byref(shape), C.byref(C.c_size_t())) == dit.DIT_ERR_UNSUPPORTED


def test_invalid_arguments_rejected_before_any_launch(dit):
    """Each call fails validation without a device; the launch counter must not move."""
    L = dit.lib()
    before = dit.dit_launch_count()
    c = dit.dit_config_klein()
    shape = dit.make_shape(1, 512, 4096, 0)
    w = dit.dit_weights()
    w.cfg = c
    fake = 0x10000  # aligned, never dereferenced: validation fails on another argument first
    # null weights / misaligned pointers / bad layer / bad batch / small workspace
    assert L.dit_dual_block_fwd(None, 0, C.byref(shape), fake, fake, fake, fake, 1 << 40, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_dual_block_fwd(C.byref(w), 0, C.byref(shape), fake + 2, fake, fake, fake, 1 << 40, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_dual_block_fwd(C.byref(w), 7, C.byref(shape), fake, fake, fake, fake, 1 << 40, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_single_block_fwd(C.byref(w), 0, C.byref(shape), fake, fake, fake, fake, 1024, None) == dit.DIT_ERR_WORKSPACE
    bad = dit.make_shape(0, 512, 4096, 0)
    assert L.dit_single_block_fwd(C.byref(w), 0, C.byref(bad), fake, fake, fake, fake, 1 << 40, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_step_fwd(C.byref(w), C.byref(shape), fake, None, fake, fake, fake, fake, fake, 1 << 40, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_modulation(C.byref(w), fake, 0, fake, fake, 1 << 20, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_rope_table(C.byref(c), fake + 4, 10, fake, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_pack_mlp_in(fake, fake + 16, 9216, 3072, None) == dit.DIT_ERR_INVALID_ARG   # overlap
    assert L.dit_pack_mlp_in(fake, fake, 100, 3072, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_pack_mlp_in(fake, fake + (1 << 40), 1 << 30, 64, None) == dit.DIT_ERR_INVALID_ARG  # 2F past limit
    assert L.dit_linear(1, 10, 48, 64, fake, fake, fake, 48, 0, None, 0, fake, 256, None) == dit.DIT_ERR_INVALID_ARG  # n % 32
    assert L.dit_linear(1, 10, 64, 60, fake, fake, fake, 64, 0, None, 0, fake, 256, None) == dit.DIT_ERR_INVALID_ARG  # k % 8
    assert L.dit_linear(1, 10, 64, 64, fake, fake, fake, 64, 1, None, 0, fake, 256, None) == dit.DIT_ERR_INVALID_ARG  # no gate
    assert L.dit_linear(1, 10, 64, 64, fake, fake, fake, 64, 0, None, 0, fake, 16, None) == dit.DIT_ERR_WORKSPACE
    big = (1 << 20) + 32  # past the token limit: rows, n_out or k
    assert L.dit_linear(1, big, 64, 64, fake, fake, fake, 64, 0, None, 0, fake, 256, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_linear(1, 10, big, 64, fake, fake, fake, big, 0, None, 0, fake, 256, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_linear(1, 10, 64, big, fake, fake, fake, 64, 0, None, 0, fake, 256, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_linear(65, 10, 64, 64, fake, fake, fake, 64, 0, None, 0, fake, 256, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_attention(1, 2, 10, fake, fake, fake, fake, 200, fake, 256, None) == dit.DIT_ERR_INVALID_ARG  # ld < 256
    assert L.dit_attention(1, 1 << 24, 10, fake, fake, fake, fake, 256, fake, 256, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_attention(1, 2, big, fake, fake, fake, fake, 256, fake, 256, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_adaln(1, 4, 300, fake, 4, 0, 0, fake, fake, fake, fake, 0, 1e-6, fake, None) == dit.DIT_ERR_UNSUPPORTED
    assert L.dit_adaln(1, 4, 256, fake, 3, 0, 0, fake, fake, fake, fake, 0, 1e-6, fake, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_adaln(1, big, 256, fake, big, 0, 0, fake, fake, fake, fake, 0, 1e-6, fake, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_adaln(65, 4, 256, fake, 4, 0, 0, fake, fake, fake, fake, 0, 1e-6, fake, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_timing_begin(0) == dit.DIT_ERR_INVALID_ARG
    assert dit.dit_launch_count() == before


def test_fp8_copies_are_validated_before_launch(dit):
    """e4m3 copies: a dual-block projection given for one stream only, a missing or
    misaligned scale, are refused before any launch (readings of the precision knob)."""
    L = dit.lib()
    before = dit.dit_launch_count()
    c = dit.dit_config_klein()
    c.n_dual, c.n_single = 1, 1
    shape = dit.make_shape(1, 512, 4096, 0)
    fake = 0x10000  # aligned, never dereferenced: the fp8 checks fail first
    dual = (dit.dit_dual_weights * 1)()
    for side in ("img", "txt"):
        sw = getattr(dual[0], side)
        for n in ("qkv", "q_norm", "k_norm", "out", "mlp_in", "mlp_out"):
            setattr(sw, n, fake)
    single = (dit.dit_single_weights * 1)()
    for n in ("qkv_mlp", "q_norm", "k_norm", "out"):
        setattr(single[0], n, fake)
    w = dit.dit_weights()
    w.cfg = c
    w.dual = C.cast(dual, C.POINTER(dit.dit_dual_weights))
    w.single = C.cast(single, C.POINTER(dit.dit_single_weights))
    d8 = (dit.dit_dual_fp8 * 1)()
    d8[0].img.qkv.q, d8[0].img.qkv.scale = fake, fake  # the text stream's copy is missing
    w.dual_fp8 = C.cast(d8, C.POINTER(dit.dit_dual_fp8))
    args = (C.byref(shape), fake, fake, fake, fake, 1 << 40, None)
    assert L.dit_dual_block_fwd(C.byref(w), 0, *args) == dit.DIT_ERR_INVALID_ARG
    d8[0].txt.qkv.q, d8[0].txt.qkv.scale = fake, fake + 4  # misaligned scale
    assert L.dit_dual_block_fwd(C.byref(w), 0, *args) == dit.DIT_ERR_INVALID_ARG
    d8[0].txt.qkv.scale = fake
    s8 = (dit.dit_single_fp8 * 1)()
    s8[0].qkv_mlp_q, s8[0].qkv_mlp_scale = fake, fake
    s8[0].out.q = fake  # out-projection copy without its scales
    w.single_fp8 = C.cast(s8, C.POINTER(dit.dit_single_fp8))
    assert L.dit_single_block_fwd(C.byref(w), 0, *args) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_step_fwd(C.byref(w), C.byref(shape), fake, None, fake, fake, fake, fake, fake, 1 << 40,
                          None) == dit.DIT_ERR_INVALID_ARG
    s8[0].qkv_mlp_q = None  # the fused projection's copy is required once single_fp8 is given
    s8[0].out.scale = fake
    assert L.dit_single_block_fwd(C.byref(w), 0, *args) == dit.DIT_ERR_INVALID_ARG
    assert dit.dit_launch_count() == before


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch, dit):
    import importlib
    mod = importlib.reload(dit)
    monkeypatch.setattr(mod, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(mod, "_lib", None)
    with pytest.raises(RuntimeError):
        mod.lib()


def test_loop_host_graph_and_helper_calls_validate_before_any_cuda_call(dit):
    """On a host without a GPU any CUDA call fails, so each of these returning its own
    validation status (not DIT_ERR_CUDA), with the launch counter unmoved, shows that the
    denoising loop, the host-buffer step, graph capture, weight quantisation, the self-test
    and the status read check their arguments before touching the device."""
    L = dit.lib()
    before = dit.dit_launch_count()
    fake = 0x10000
    c = dit.dit_config_klein()
    c.n_dual, c.n_single = 0, 0
    w = dit.dit_weights()
    w.cfg = c
    w.mod.t_in = w.mod.t_out = w.mod.mod = fake
    w.x_emb = w.ctx_emb = w.proj_out = fake
    shape = dit.make_shape(1, 512, 4096, 0)
    ref_shape = dit.make_shape(1, 512, 4096, 1024)
    big = 1 << 40
    sig = (C.c_float * 9)(*([0.9, 0.7, 0.5, 0.2, 0.0] + [0.0] * 4))
    bad_sig = (C.c_float * 9)(*([0.9, 1500.0, 0.5, 0.2, 0.0] + [0.0] * 4))
    INV, WS = dit.DIT_ERR_INVALID_ARG, dit.DIT_ERR_WORKSPACE
    den = lambda sh, ref, sg, steps, nbytes: L.dit_denoise_fwd(C.byref(w), C.byref(sh), fake, ref, fake, fake, sg,
                                                               steps, fake, nbytes, None)
    assert den(shape, None, sig, 0, big) == INV            # at least one step
    assert den(shape, None, sig, 9, big) == INV            # at most eight
    assert den(shape, None, bad_sig, 4, big) == INV        # sigma outside [0, 1000]
    assert den(shape, None, None, 4, big) == INV           # no schedule
    assert den(ref_shape, None, sig, 4, big) == INV        # reference rows without reference tokens
    assert den(shape, fake, sig, 4, big) == INV            # reference tokens without reference rows
    assert den(shape, None, sig, 4, 4096) == WS
    host = lambda sh, ref, nbytes: L.dit_step_host(C.byref(w), C.byref(sh), fake, ref, fake, fake, fake, fake, fake,
                                                   nbytes, None)
    assert host(ref_shape, None, big) == INV
    assert host(shape, None, 4096) == WS
    assert L.dit_step_host(C.byref(w), C.byref(shape), None, None, fake, fake, fake, fake, fake, big, None) == INV
    g = C.c_void_p(123)
    assert L.dit_step_graph_create(C.byref(w), C.byref(shape), fake, None, fake, fake, fake, fake, fake, 4096, 0, None,
                                   C.byref(g)) == WS
    assert g.value is None                                  # no graph handle on failure
    assert L.dit_step_graph_create(C.byref(w), C.byref(shape), fake, None, fake, fake, fake, fake, fake, big, 0, None,
                                   None) == INV
    assert L.dit_graph_launch(None, None) == INV
    assert L.dit_graph_destroy(None) == dit.DIT_OK
    assert L.dit_quantize_rows_fp8(fake, 4, 24, fake, fake, None) == INV       # cols % 16
    assert L.dit_quantize_rows_fp8(fake, 4, 32, fake, fake + 4, None) == INV   # misaligned scales
    assert L.dit_quantize_rows_fp8(fake, 0, 32, fake, fake, None) == INV
    assert L.dit_quantize_rows_fp8(fake, (1 << 20) + 1, 32, fake, fake, None) == INV
    assert L.dit_quantize_rows_fp8(fake, 4, (1 << 20) + 16, fake, fake, None) == INV
    assert L.dit_selftest_wait_timeout(fake, 256, 0, None) == INV
    assert L.dit_selftest_wait_timeout(fake, 256, 2000000, None) == INV
    assert L.dit_selftest_wait_timeout(fake, 8, 100, None) == INV
    assert L.dit_sync_status(None, None, None) == INV
    assert L.dit_sync_status(fake + 8, None, None) == INV
    assert dit.dit_launch_count() == before


def test_header_is_plain_c_and_host_entry_points_work_from_c(dit, tmp_path):
    """tests/c/abi_from_c.c, compiled as C11 with warnings as errors against include/dit.h
    and linked to libdit.so: the header needs no C++ or CUDA header, and the host-side
    calls (klein config, workspace sizes, token ids, refusals before any launch) behave
    as documented when called from C."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    pkg = os.path.dirname(dit.LIB_PATH)
    exe = str(tmp_path / "abi_from_c")
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_from_c.c"), "-L", pkg, "-ldit", f"-Wl,-rpath,{pkg}",
                    "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr
