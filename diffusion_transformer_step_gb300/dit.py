"""Thin Python binding of the C ABI in include/dit.h (ctypes).

Argument marshalling only: every function here forwards to the function of the same
name in libdit.so, passing device pointers (``tensor.data_ptr()``), sizes and the CUDA
stream handle; all device work runs in the library's kernels.  PyTorch is used only to
own device memory and streams.  There is no fallback: if the library is not built, or a
call returns an error status, a ``DitError`` is raised.
"""
from __future__ import annotations

import ctypes as C
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdit.so")

DIT_OK, DIT_ERR_INVALID_ARG, DIT_ERR_UNSUPPORTED, DIT_ERR_WORKSPACE, DIT_ERR_CUDA, DIT_ERR_TIMEOUT = range(6)
DIT_EPI_STORE, DIT_EPI_GATED_RESIDUAL, DIT_EPI_SWIGLU = range(3)


class DitError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


class dit_config(C.Structure):
    _fields_ = [("hidden", C.c_int), ("heads", C.c_int), ("head_dim", C.c_int), ("mlp_hidden", C.c_int),
                ("n_dual", C.c_int), ("n_single", C.c_int), ("in_channels", C.c_int), ("txt_dim", C.c_int),
                ("rope_theta", C.c_float), ("axes_dim", C.c_int * 4), ("eps", C.c_float)]


class dit_shape(C.Structure):
    _fields_ = [("batch", C.c_int), ("n_txt", C.c_int), ("n_img", C.c_int), ("n_ref", C.c_int)]


class dit_mod_weights(C.Structure):
    _fields_ = [("t_in", C.c_void_p), ("t_out", C.c_void_p), ("mod", C.c_void_p)]


class dit_stream_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("qkv", "q_norm", "k_norm", "out", "mlp_in", "mlp_out")]


class dit_dual_weights(C.Structure):
    _fields_ = [("img", dit_stream_weights), ("txt", dit_stream_weights)]


class dit_single_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("qkv_mlp", "q_norm", "k_norm", "out")]


class dit_fp8_matrix(C.Structure):
    _fields_ = [("q", C.c_void_p), ("scale", C.c_void_p)]


class dit_single_fp8(C.Structure):
    _fields_ = [("qkv_mlp_q", C.c_void_p), ("qkv_mlp_scale", C.c_void_p), ("out", dit_fp8_matrix)]


class dit_stream_fp8(C.Structure):
    _fields_ = [(n, dit_fp8_matrix) for n in ("qkv", "mlp_in", "out", "mlp_out")]


class dit_dual_fp8(C.Structure):
    _fields_ = [("img", dit_stream_fp8), ("txt", dit_stream_fp8)]


class dit_weights(C.Structure):
    _fields_ = [("cfg", dit_config), ("mod", dit_mod_weights), ("x_emb", C.c_void_p), ("ctx_emb", C.c_void_p),
                ("proj_out", C.c_void_p), ("dual", C.POINTER(dit_dual_weights)),
                ("single", C.POINTER(dit_single_weights)), ("single_fp8", C.POINTER(dit_single_fp8)),
                ("dual_fp8", C.POINTER(dit_dual_fp8))]


_P = C.c_void_p
_I = C.c_int
_SZ = C.c_size_t
_LL = C.c_longlong
_F = C.c_float

# name -> (restype, argtypes)
_SIGS = {
    "dit_status_string": (C.c_char_p, [_I]),
    "dit_config_klein": (_I, [C.POINTER(dit_config)]),
    "dit_workspace_size": (_I, [C.POINTER(dit_config), C.POINTER(dit_shape), C.POINTER(_SZ)]),
    "dit_token_ids": (_I, [C.POINTER(dit_shape), _I, _I, C.POINTER(_I), _I, _P]),
    "dit_rope_table": (_I, [C.POINTER(dit_config), _P, _I, _P, _P]),
    "dit_pack_mlp_in": (_I, [_P, _P, _I, _I, _P]),
    "dit_quantize_rows_fp8": (_I, [_P, _I, _I, _P, _P, _P]),
    "dit_modulation": (_I, [C.POINTER(dit_weights), _P, _I, _P, _P, _SZ, _P]),
    "dit_dual_block_fwd": (_I, [C.POINTER(dit_weights), _I, C.POINTER(dit_shape), _P, _P, _P, _P, _SZ, _P]),
    "dit_single_block_fwd": (_I, [C.POINTER(dit_weights), _I, C.POINTER(dit_shape), _P, _P, _P, _P, _SZ, _P]),
    "dit_step_fwd": (_I, [C.POINTER(dit_weights), C.POINTER(dit_shape), _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "dit_denoise_fwd": (_I, [C.POINTER(dit_weights), C.POINTER(dit_shape), _P, _P, _P, _P, C.POINTER(_F), _I, _P,
                             _SZ, _P]),
    "dit_step_host": (_I, [C.POINTER(dit_weights), C.POINTER(dit_shape), _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "dit_sync_status": (_I, [_P, _P, C.POINTER(C.c_uint32)]),
    "dit_adaln": (_I, [_I, _I, _I, _P, _I, _I, _I, _P, _P, _P, _P, _LL, _F, _P, _P]),
    "dit_linear": (_I, [_I, _I, _I, _I, _P, _P, _P, _I, _I, _P, _LL, _P, _SZ, _P]),
    "dit_attention": (_I, [_I, _I, _I, _P, _P, _P, _P, _I, _P, _SZ, _P]),
    "dit_modulation_static": (_I, [C.POINTER(dit_weights), _P, _I, _P, _P]),
    "dit_step_graph_create": (_I, [C.POINTER(dit_weights), C.POINTER(dit_shape), _P, _P, _P, _P, _P, _P, _P, _SZ,
                                   _I, _P, C.POINTER(_P)]),
    "dit_graph_launch": (_I, [_P, _P]),
    "dit_graph_destroy": (_I, [_P]),
    "dit_selftest_wait_timeout": (_I, [_P, _SZ, C.c_uint, _P]),
    "dit_launch_count": (C.c_ulonglong, []),
    "dit_timing_begin": (_I, [_I]),
    "dit_timing_select": (_I, [C.c_uint]),
    "dit_timing_end": (_I, [C.POINTER(_I), C.POINTER(_I), C.POINTER(_F), _I]),
    "dit_kernel_class_name": (C.c_char_p, [_I]),
}

_lib = None


def lib():
    """Load libdit.so (built in-tree by the package's build step).  Raises if missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run `python -c \"import __graft_entry__ as g; g.build()\"`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(fn, st):
    if st != DIT_OK:
        raise DitError(fn, st, lib().dit_status_string(st).decode())


def _ptr(t):
    """Device or host pointer of a tensor (or None / int passthrough)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_config(hidden=3072, heads=24, head_dim=128, mlp_hidden=9216, n_dual=5, n_single=20, in_channels=128,
                txt_dim=7680, rope_theta=2000.0, axes_dim=(32, 32, 32, 32), eps=1e-6) -> dit_config:
    c = dit_config()
    c.hidden, c.heads, c.head_dim, c.mlp_hidden = hidden, heads, head_dim, mlp_hidden
    c.n_dual, c.n_single, c.in_channels, c.txt_dim = n_dual, n_single, in_channels, txt_dim
    c.rope_theta = rope_theta
    for i in range(4):
        c.axes_dim[i] = axes_dim[i]
    c.eps = eps
    return c


def make_shape(batch, n_txt, n_img, n_ref=0) -> dit_shape:
    s = dit_shape()
    s.batch, s.n_txt, s.n_img, s.n_ref = batch, n_txt, n_img, n_ref
    return s


# ---------------------------------------------------------------------------------- calls
def dit_status_string(st: int) -> str:
    return lib().dit_status_string(st).decode()


def dit_config_klein() -> dit_config:
    c = dit_config()
    _check("dit_config_klein", lib().dit_config_klein(C.byref(c)))
    return c


def dit_workspace_size(cfg: dit_config, shape: dit_shape) -> int:
    n = _SZ(0)
    _check("dit_workspace_size", lib().dit_workspace_size(C.byref(cfg), C.byref(shape), C.byref(n)))
    return n.value


def dit_token_ids(shape: dit_shape, grid_h: int, grid_w: int, ref_grids=()):
    """Returns an int32 CPU tensor [N, 4] of (t, h, w, l) ids, built by the library."""
    import torch
    N = shape.n_txt + shape.n_img + shape.n_ref
    ids = torch.empty((N, 4), dtype=torch.int32)
    flat = [int(v) for g in ref_grids for v in g]
    arr = (C.c_int * max(1, len(flat)))(*flat) if flat else None
    _check("dit_token_ids", lib().dit_token_ids(C.byref(shape), grid_h, grid_w, arr, len(ref_grids), ids.data_ptr()))
    return ids


def dit_rope_table(cfg: dit_config, ids_dev, n: int, table_dev, stream=None):
    _check("dit_rope_table", lib().dit_rope_table(C.byref(cfg), _ptr(ids_dev), n, _ptr(table_dev), _stream(stream)))


def dit_pack_mlp_in(src_dev, dst_dev, mlp_hidden: int, cols: int, stream=None):
    _check("dit_pack_mlp_in", lib().dit_pack_mlp_in(_ptr(src_dev), _ptr(dst_dev), mlp_hidden, cols, _stream(stream)))


def dit_quantize_rows_fp8(w_dev, rows: int, cols: int, q_dev, scale_dev, stream=None):
    _check("dit_quantize_rows_fp8", lib().dit_quantize_rows_fp8(_ptr(w_dev), rows, cols, _ptr(q_dev), _ptr(scale_dev),
                                                                 _stream(stream)))


def dit_modulation(w: dit_weights, sigma_dev, batch: int, mod_dev, ws, ws_bytes: int, stream=None):
    _check("dit_modulation", lib().dit_modulation(C.byref(w), _ptr(sigma_dev), batch, _ptr(mod_dev), _ptr(ws),
                                                   ws_bytes, _stream(stream)))


def dit_dual_block_fwd(w: dit_weights, layer: int, shape: dit_shape, x_dev, mod_dev, rope_dev, ws, ws_bytes: int,
                       stream=None):
    _check("dit_dual_block_fwd", lib().dit_dual_block_fwd(C.byref(w), layer, C.byref(shape), _ptr(x_dev), _ptr(mod_dev),
                                                           _ptr(rope_dev), _ptr(ws), ws_bytes, _stream(stream)))


def dit_single_block_fwd(w: dit_weights, layer: int, shape: dit_shape, x_dev, mod_dev, rope_dev, ws, ws_bytes: int,
                         stream=None):
    _check("dit_single_block_fwd", lib().dit_single_block_fwd(C.byref(w), layer, C.byref(shape), _ptr(x_dev),
                                                               _ptr(mod_dev), _ptr(rope_dev), _ptr(ws), ws_bytes,
                                                               _stream(stream)))


def dit_step_fwd(w: dit_weights, shape: dit_shape, img_tokens, ref_tokens, txt_emb, rope_dev, sigma_dev, velocity_out,
                 ws, ws_bytes: int, stream=None):
    _check("dit_step_fwd", lib().dit_step_fwd(C.byref(w), C.byref(shape), _ptr(img_tokens), _ptr(ref_tokens),
                                               _ptr(txt_emb), _ptr(rope_dev), _ptr(sigma_dev), _ptr(velocity_out),
                                               _ptr(ws), ws_bytes, _stream(stream)))


def dit_denoise_fwd(w: dit_weights, shape: dit_shape, x_tokens, ref_tokens, txt_emb, rope_dev, sigmas, ws,
                    ws_bytes: int, stream=None):
    """The steps-long Euler loop on the device, in place on x_tokens; `sigmas` is a host
    sequence of steps + 1 floats."""
    arr = (_F * len(sigmas))(*[float(v) for v in sigmas])
    _check("dit_denoise_fwd", lib().dit_denoise_fwd(C.byref(w), C.byref(shape), _ptr(x_tokens), _ptr(ref_tokens),
                                                     _ptr(txt_emb), _ptr(rope_dev), arr, len(sigmas) - 1, _ptr(ws),
                                                     ws_bytes, _stream(stream)))


def dit_step_host(w: dit_weights, shape: dit_shape, img_tokens_host, ref_tokens_host, txt_emb_host, rope_dev,
                  sigma_host, velocity_host, ws, ws_bytes: int, stream=None):
    _check("dit_step_host", lib().dit_step_host(C.byref(w), C.byref(shape), _ptr(img_tokens_host),
                                                 _ptr(ref_tokens_host), _ptr(txt_emb_host), _ptr(rope_dev),
                                                 _ptr(sigma_host), _ptr(velocity_host), _ptr(ws), ws_bytes,
                                                 _stream(stream)))


def dit_step_graph_create(w: dit_weights, shape: dit_shape, img_tokens, ref_tokens, txt_emb, rope_dev, sigma,
                          velocity_out, ws, ws_bytes: int, host_io: bool = False, stream=None) -> int:
    """Capture one dit_step_fwd (host_io False) or dit_step_host (host_io True) call into a
    CUDA graph; returns the opaque handle (an int)."""
    h = _P()
    _check("dit_step_graph_create", lib().dit_step_graph_create(
        C.byref(w), C.byref(shape), _ptr(img_tokens), _ptr(ref_tokens), _ptr(txt_emb), _ptr(rope_dev), _ptr(sigma),
        _ptr(velocity_out), _ptr(ws), ws_bytes, 1 if host_io else 0, _stream(stream), C.byref(h)))
    return h.value


def dit_graph_launch(graph: int, stream=None):
    _check("dit_graph_launch", lib().dit_graph_launch(graph, _stream(stream)))


def dit_graph_destroy(graph: int):
    _check("dit_graph_destroy", lib().dit_graph_destroy(graph))


def dit_sync_status(ws, stream=None):
    """Returns (status, where).  Does not raise on DIT_ERR_TIMEOUT."""
    where = C.c_uint32(0)
    st = lib().dit_sync_status(_ptr(ws), _stream(stream), C.byref(where))
    if st not in (DIT_OK, DIT_ERR_TIMEOUT):
        _check("dit_sync_status", st)
    return st, where.value


def dit_adaln(batch, rows, hidden, x_dev, x_rows, x_row0, split, shift_lo, scale_lo, shift_hi, scale_hi, mod_stride,
              eps, y_dev, stream=None):
    _check("dit_adaln", lib().dit_adaln(batch, rows, hidden, _ptr(x_dev), x_rows, x_row0, split, _ptr(shift_lo),
                                         _ptr(scale_lo), _ptr(shift_hi), _ptr(scale_hi), mod_stride, eps, _ptr(y_dev),
                                         _stream(stream)))


def dit_linear(batch, rows, n_out, k, a_dev, w_dev, out_dev, ld_out, epi, gate_dev, gate_stride, ws, ws_bytes,
               stream=None):
    _check("dit_linear", lib().dit_linear(batch, rows, n_out, k, _ptr(a_dev), _ptr(w_dev), _ptr(out_dev), ld_out, epi,
                                           _ptr(gate_dev), gate_stride, _ptr(ws), ws_bytes, _stream(stream)))


def dit_attention(batch, heads, n, q_dev, k_dev, v_dev, out_dev, ld_out, ws, ws_bytes, stream=None):
    _check("dit_attention", lib().dit_attention(batch, heads, n, _ptr(q_dev), _ptr(k_dev), _ptr(v_dev), _ptr(out_dev),
                                                 ld_out, _ptr(ws), ws_bytes, _stream(stream)))


def dit_modulation_static(w: dit_weights, sigma_dev, batch: int, mod_dev, stream=None):
    """dit_modulation without a workspace (scratch in a fixed device array of the library;
    batch <= 8, hidden <= 4096), for callers that cannot allocate device memory."""
    _check("dit_modulation_static", lib().dit_modulation_static(C.byref(w), _ptr(sigma_dev), batch, _ptr(mod_dev),
                                                                 _stream(stream)))


def dit_selftest_wait_timeout(ws, ws_bytes: int, limit_us: int, stream=None):
    """Launch the bounded-wait self-test kernel (a wait that can never complete)."""
    _check("dit_selftest_wait_timeout", lib().dit_selftest_wait_timeout(_ptr(ws), ws_bytes, limit_us, _stream(stream)))


def dit_launch_count() -> int:
    return int(lib().dit_launch_count())


def dit_timing_begin(max_records: int):
    _check("dit_timing_begin", lib().dit_timing_begin(max_records))


def dit_timing_select(class_mask: int):
    _check("dit_timing_select", lib().dit_timing_select(class_mask & 0xFFFFFFFF))


def dit_timing_end(cap: int):
    """Returns a list of (kernel class name, ms) per recorded launch."""
    n = _I(0)
    cls = (_I * max(cap, 1))()
    ms = (_F * max(cap, 1))()
    _check("dit_timing_end", lib().dit_timing_end(C.byref(n), cls, ms, cap))
    return [(lib().dit_kernel_class_name(cls[i]).decode(), float(ms[i])) for i in range(n.value)]


def dit_kernel_class_name(cls: int) -> str:
    return lib().dit_kernel_class_name(cls).decode()


# ---------------------------------------------------------------------------------- weights
class DeviceWeights:
    """Device copies of a model's weights in the library's layouts, and the dit_weights
    struct that points at them.  ``logical`` is a dict as produced by
    ``synth.model_weights`` (logical layouts: MLP-in rows [gate; up]); MLP-in weights are
    rearranged on the device by dit_pack_mlp_in.  Keeps every tensor alive."""

    def __init__(self, widths, logical: dict, device="cuda", n_dual=None, n_single=None, fp8=False):
        import torch
        self.widths = widths
        H, F = widths.hidden, widths.mlp_hidden
        nd = len(logical.get("dual", [])) if n_dual is None else n_dual
        ns = len(logical.get("single", [])) if n_single is None else n_single
        self.cfg = make_config(hidden=H, heads=widths.heads, head_dim=widths.head_dim, mlp_hidden=F, n_dual=nd,
                               n_single=ns, in_channels=widths.in_channels, txt_dim=widths.txt_dim)
        keep = []

        def dev(t):
            d = t.to(device=device, dtype=torch.bfloat16).contiguous()
            keep.append(d)
            return d

        def packed(t, rows_before=0):
            src = t.to(device=device, dtype=torch.bfloat16).contiguous()  # temporary, logical order
            dst = torch.empty_like(src)
            if rows_before:
                dst[:rows_before].copy_(src[:rows_before])
            dit_pack_mlp_in(src[rows_before:], dst[rows_before:], F, src.shape[1])
            keep.append(dst)
            return dst

        w = dit_weights()
        w.cfg = self.cfg
        # block-level users may pass only the blocks; absent tensors stay NULL
        m = logical.get("mod")
        if m is not None:
            w.mod.t_in, w.mod.t_out, w.mod.mod = (dev(m[k]).data_ptr() for k in ("t_in", "t_out", "mod"))
        for key in ("x_emb", "ctx_emb", "proj_out"):
            if logical.get(key) is not None:
                setattr(w, key, dev(logical[key]).data_ptr())
        self._dual = (dit_dual_weights * max(1, nd))()
        for i in range(nd):
            for side, src in (("img", logical["dual"][i][0]), ("txt", logical["dual"][i][1])):
                sw = getattr(self._dual[i], side)
                sw.qkv = dev(src["qkv"]).data_ptr()
                sw.q_norm = dev(src["q_norm"]).data_ptr()
                sw.k_norm = dev(src["k_norm"]).data_ptr()
                sw.out = dev(src["out"]).data_ptr()
                sw.mlp_in = packed(src["mlp_in"]).data_ptr()
                sw.mlp_out = dev(src["mlp_out"]).data_ptr()
        self._single = (dit_single_weights * max(1, ns))()
        for i in range(ns):
            src = logical["single"][i]
            s = self._single[i]
            s.qkv_mlp = packed(src["qkv_mlp"], rows_before=3 * H).data_ptr()
            s.q_norm = dev(src["q_norm"]).data_ptr()
            s.k_norm = dev(src["k_norm"]).data_ptr()
            s.out = dev(src["out"]).data_ptr()
        w.dual = C.cast(self._dual, C.POINTER(dit_dual_weights))
        w.single = C.cast(self._single, C.POINTER(dit_single_weights))
        # e4m3 copies (the library's reading of the precision knob): fp8="fused" quantises only
        # the single-stream fused QKV + MLP-in projections; fp8=True or "all" every block
        # projection (dual QKV / MLP-in / out / MLP-out, single fused / out).
        scope = {False: None, None: None, True: "all", "all": "all", "fused": "fused"}[fp8]

        def quant(ptr, rows, cols):
            q = torch.empty((rows, cols), dtype=torch.uint8, device=device)
            sc = torch.empty((rows,), dtype=torch.float32, device=device)
            dit_quantize_rows_fp8(ptr, rows, cols, q, sc)
            keep.extend([q, sc])
            return q.data_ptr(), sc.data_ptr()

        if scope and ns > 0:
            self._single_fp8 = (dit_single_fp8 * ns)()
            for i in range(ns):
                f8 = self._single_fp8[i]
                f8.qkv_mlp_q, f8.qkv_mlp_scale = quant(self._single[i].qkv_mlp, 3 * H + 2 * F, H)
                if scope == "all":
                    f8.out.q, f8.out.scale = quant(self._single[i].out, H, H + F)
            w.single_fp8 = C.cast(self._single_fp8, C.POINTER(dit_single_fp8))
        if scope == "all" and nd > 0:
            self._dual_fp8 = (dit_dual_fp8 * nd)()
            for i in range(nd):
                for side in ("img", "txt"):
                    sw, f8 = getattr(self._dual[i], side), getattr(self._dual_fp8[i], side)
                    f8.qkv.q, f8.qkv.scale = quant(sw.qkv, 3 * H, H)
                    f8.mlp_in.q, f8.mlp_in.scale = quant(sw.mlp_in, 2 * F, H)
                    f8.out.q, f8.out.scale = quant(sw.out, H, H)
                    f8.mlp_out.q, f8.mlp_out.scale = quant(sw.mlp_out, H, F)
            w.dual_fp8 = C.cast(self._dual_fp8, C.POINTER(dit_dual_fp8))
        self.w = w
        self._keep = keep
        torch.cuda.synchronize()
