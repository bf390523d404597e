"""Thin ctypes binding of libacnn (include/acnn.h).

Two layers, both pure argument marshalling -- every step of the computation
runs in the library's CUDA kernels:

* ``acnn_*`` functions with the C names and arguments (pointers as ints or
  tensors, sizes as ints), returning the int status;
* tensor-level helpers (``conv2d_fused``, ``pool2d``, ...) that allocate the
  output with PyTorch, pass raw device pointers and the current stream, and
  raise ``AcnnError`` on a non-zero status.

The library is loaded from ``activation_cnn_gb300/lib/libacnn.so``; if it is
missing the first call raises -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .inputs import NHWC, NCHW, F32, F16, BF16, TORCH_DTYPE  # noqa: F401  (enum values)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libacnn.so")

ACT_NONE, ACT_RELU, ACT_SILU, ACT_PRELU = 0, 1, 2, 3
RES_NONE, RES_ADD_THEN_ACT, RES_ACT_THEN_ADD = 0, 1, 2
POOL_MAX, POOL_AVG = 0, 1
RESIZE_NEAREST, RESIZE_BILINEAR = 0, 1

STATUS = {
    0: "ACNN_OK", 1: "ACNN_ERR_NULL_POINTER", 2: "ACNN_ERR_BAD_GEOMETRY",
    3: "ACNN_ERR_UNSUPPORTED", 4: "ACNN_ERR_MISALIGNED", 5: "ACNN_ERR_WORKSPACE",
    6: "ACNN_ERR_ALIAS", 7: "ACNN_ERR_BAD_ENUM", 8: "ACNN_ERR_CUDA",
    9: "ACNN_ERR_DEVICE_TIMEOUT", 10: "ACNN_ERR_TOO_LARGE",
}
EXPORTS = (
    "acnn_conv2d_fused", "acnn_conv2d_out_hw", "acnn_conv2d_workspace_size", "acnn_conv2d_path",
    "acnn_pool2d", "acnn_resize2d", "acnn_concat", "acnn_deconv2d", "acnn_frame_prep_quarter",
    "acnn_frame_flow_out", "acnn_frame_refine_prep", "acnn_frame_refine_out", "acnn_film",
    "acnn_conv2d_prepacked_size", "acnn_conv2d_prepack", "acnn_conv2d_prepacked_workspace_size",
    "acnn_conv2d_fused_prepacked",
    "acnn_status_string", "acnn_last_device_status", "acnn_set_wait_budget",
    "acnn_section_begin", "acnn_section_end", "acnn_section_launch", "acnn_section_destroy",
    "acnn_device_sm_count", "acnn_conv2d_fused_noalloc", "acnn_conv2d_plan",
    "acnn_conv2d_fused_cat2", "acnn_conv2d_force_plan", "acnn_conv2d_force_path",
    "acnn_conv2d_fused_pool2", "acnn_conv2d_fused_up2", "acnn_deconv2d_workspace_size",
    "acnn_deconv2d_ws", "acnn_conv2d_fused_prepacked_staged",
)
NOALLOC_SCRATCH_BYTES = 16 << 20  # ACNN_NOALLOC_SCRATCH_BYTES in include/acnn.h


class AcnnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status_string(status)})")


class ConvDesc(ctypes.Structure):
    _fields_ = [(k, ctypes.c_int) for k in
                ("n", "h", "w", "c_in", "c_out", "kh", "kw", "stride", "pad", "layout", "dtype")]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int


def lib() -> ctypes.CDLL:
    """Load libacnn.so (raises if it was not built: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libacnn.so not found at {LIB_PATH}; build it with "
                               "`python -m activation_cnn_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        D = ctypes.POINTER(ConvDesc)
        L.acnn_conv2d_fused.argtypes = [D, _P, _P, _P, _P, _P, _I, _I, _P, _P, ctypes.c_size_t, _P]
        L.acnn_conv2d_out_hw.argtypes = [D, ctypes.POINTER(_I), ctypes.POINTER(_I)]
        L.acnn_conv2d_fused_cat2.argtypes = [D, _P, _I, _P, _P, _P, _P, _P, _I, _I, _P, _P,
                                             ctypes.c_size_t, _P]
        L.acnn_conv2d_workspace_size.argtypes = [D]
        L.acnn_conv2d_workspace_size.restype = ctypes.c_size_t
        L.acnn_conv2d_prepacked_size.argtypes = [D]
        L.acnn_conv2d_prepacked_size.restype = ctypes.c_size_t
        L.acnn_conv2d_prepacked_workspace_size.argtypes = [D]
        L.acnn_conv2d_prepacked_workspace_size.restype = ctypes.c_size_t
        L.acnn_conv2d_prepack.argtypes = [D, _P, _P, _P]
        L.acnn_conv2d_fused_prepacked.argtypes = [D, _P, _P, _P, _P, _P, _I, _I, _P, _P,
                                                  ctypes.c_size_t, _P]
        L.acnn_conv2d_path.argtypes = [D]
        L.acnn_pool2d.argtypes = [_I] * 10 + [_P, _P, _P]
        L.acnn_resize2d.argtypes = [_I] * 10 + [_P, _P, _P]
        L.acnn_concat.argtypes = [_I] * 7 + [_P, _P, _P, _P]
        L.acnn_deconv2d.argtypes = [D, _P, _P, _P, _P, _I, _I, _P, _P]
        L.acnn_frame_prep_quarter.argtypes = [_I, _I, _P, _P, ctypes.c_float, _I, _P, _P]
        L.acnn_frame_flow_out.argtypes = [_I, _I, _P, _I, _P, _P, _P, _P, _P]
        L.acnn_frame_refine_prep.argtypes = [_I, _I, _P, _I, _P, _P, _I, _P, _P]
        L.acnn_frame_refine_out.argtypes = [_I, _I, _I, _P, _I, _P, _P, _P, _P]
        L.acnn_film.argtypes = [_I, ctypes.c_longlong, _I, _P, ctypes.c_float, _P, _P, _I, _P, _P,
                                _P, _P]
        L.acnn_status_string.argtypes = [_I]
        L.acnn_status_string.restype = ctypes.c_char_p
        L.acnn_last_device_status.argtypes = [_P]
        L.acnn_set_wait_budget.argtypes = [ctypes.c_longlong]
        L.acnn_section_begin.argtypes = [_P]
        L.acnn_section_end.argtypes = [_P, ctypes.POINTER(_P)]
        L.acnn_section_launch.argtypes = [_P, _P]
        L.acnn_section_destroy.argtypes = [_P]
        L.acnn_device_sm_count.argtypes = []
        L.acnn_conv2d_fused_noalloc.argtypes = [D, _P, _P, _P, _P, _P, _I, _I, _P, _P]
        L.acnn_conv2d_plan.argtypes = [D, ctypes.c_size_t] + [ctypes.POINTER(_I)] * 3
        L.acnn_conv2d_force_plan.argtypes = [_I, _I, _I]
        L.acnn_conv2d_fused_pool2.argtypes = [D, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P]
        L.acnn_conv2d_fused_prepacked_staged.argtypes = [D, _P, _P, _P, _P, _P, _P, _I, _I, _P,
                                                         _P, _P, ctypes.c_size_t, _P]
        L.acnn_deconv2d_workspace_size.argtypes = [D, _I]
        L.acnn_deconv2d_workspace_size.restype = ctypes.c_size_t
        L.acnn_deconv2d_ws.argtypes = [D, _P, _P, _P, _P, _I, _I, _P, _P, ctypes.c_size_t, _P]
        L.acnn_conv2d_fused_up2.argtypes = [D, _P, _I, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P,
                                            ctypes.c_size_t, _P]
        L.acnn_conv2d_force_path.argtypes = [_I, _I]
        _lib = L
    return _lib


# ------------------------------------------------------------------ raw ABI
def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def status_string(status: int) -> str:
    return lib().acnn_status_string(status).decode()


def acnn_conv2d_fused(desc, x, w, bias, alpha, residual, res_mode, act, y, workspace, ws_bytes,
                      stream=None) -> int:
    return lib().acnn_conv2d_fused(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias), _ptr(alpha),
                                   _ptr(residual), res_mode, act, _ptr(y), _ptr(workspace),
                                   ws_bytes, _stream(stream))


def acnn_conv2d_fused_noalloc(desc, x, w, bias, alpha, residual, res_mode, act, y,
                              stream=None) -> int:
    """conv2d_fused for callers that cannot allocate: scratch comes from a static
    device array inside the library (see include/acnn.h)."""
    return lib().acnn_conv2d_fused_noalloc(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias),
                                           _ptr(alpha), _ptr(residual), res_mode, act, _ptr(y),
                                           _stream(stream))


def acnn_conv2d_out_hw(desc):
    oh, ow = _I(), _I()
    st = lib().acnn_conv2d_out_hw(ctypes.byref(desc), ctypes.byref(oh), ctypes.byref(ow))
    return st, oh.value, ow.value


def acnn_conv2d_workspace_size(desc) -> int:
    return lib().acnn_conv2d_workspace_size(ctypes.byref(desc))


def acnn_conv2d_prepacked_size(desc) -> int:
    return lib().acnn_conv2d_prepacked_size(ctypes.byref(desc))


def acnn_conv2d_prepacked_workspace_size(desc) -> int:
    return lib().acnn_conv2d_prepacked_workspace_size(ctypes.byref(desc))


def acnn_conv2d_prepack(desc, w, w_packed, stream=None) -> int:
    return lib().acnn_conv2d_prepack(ctypes.byref(desc), _ptr(w), _ptr(w_packed),
                                     _stream(stream))


def acnn_conv2d_fused_prepacked(desc, x, w_packed, bias, alpha, residual, res_mode, act, y,
                                workspace, ws_bytes, stream=None) -> int:
    return lib().acnn_conv2d_fused_prepacked(ctypes.byref(desc), _ptr(x), _ptr(w_packed),
                                             _ptr(bias), _ptr(alpha), _ptr(residual), res_mode,
                                             act, _ptr(y), _ptr(workspace), ws_bytes,
                                             _stream(stream))


def acnn_conv2d_plan(desc, ws_bytes):
    """(status, rows, bn, splits) of the tensor-core plan with ws_bytes of workspace."""
    rows, bn, sp = _I(), _I(), _I()
    st = lib().acnn_conv2d_plan(ctypes.byref(desc), ws_bytes, ctypes.byref(rows),
                                ctypes.byref(bn), ctypes.byref(sp))
    return st, rows.value, bn.value, sp.value


def acnn_conv2d_force_plan(bn: int, rows: int = 128, splits: int = 1) -> int:
    return lib().acnn_conv2d_force_plan(bn, rows, splits)


def acnn_conv2d_force_path(path: int, variant: int = 0) -> int:
    return lib().acnn_conv2d_force_path(path, variant)


def acnn_conv2d_path(desc) -> int:
    return lib().acnn_conv2d_path(ctypes.byref(desc))


def acnn_pool2d(kind, n, h, w, c, k, stride, pad, layout, dtype, x, y, stream=None) -> int:
    return lib().acnn_pool2d(kind, n, h, w, c, k, stride, pad, layout, dtype, _ptr(x), _ptr(y),
                             _stream(stream))


def acnn_resize2d(mode, n, c, h, w, oh, ow, layout, in_dtype, out_dtype, x, y,
                  stream=None) -> int:
    return lib().acnn_resize2d(mode, n, c, h, w, oh, ow, layout, in_dtype, out_dtype, _ptr(x),
                               _ptr(y), _stream(stream))


def acnn_concat(n, h, w, c_a, c_b, layout, dtype, a, b, y, stream=None) -> int:
    return lib().acnn_concat(n, h, w, c_a, c_b, layout, dtype, _ptr(a), _ptr(b), _ptr(y),
                             _stream(stream))


def acnn_deconv2d(desc, x, w, bias, alpha, act, out_dtype, y, stream=None) -> int:
    return lib().acnn_deconv2d(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias), _ptr(alpha),
                               act, out_dtype, _ptr(y), _stream(stream))


def acnn_frame_prep_quarter(h, w, rgba0, rgba1, t, out_dtype, y, stream=None) -> int:
    return lib().acnn_frame_prep_quarter(h, w, _ptr(rgba0), _ptr(rgba1), float(t), out_dtype,
                                         _ptr(y), _stream(stream))


def acnn_frame_flow_out(h, w, tmp8, tmp8_dtype, rgba0, rgba1, refine_res, out,
                        stream=None) -> int:
    return lib().acnn_frame_flow_out(h, w, _ptr(tmp8), tmp8_dtype, _ptr(rgba0), _ptr(rgba1),
                                     _ptr(refine_res), _ptr(out), _stream(stream))


def acnn_frame_refine_prep(h, w, tmp8, tmp8_dtype, rgba0, rgba1, out_dtype, y,
                           stream=None) -> int:
    return lib().acnn_frame_refine_prep(h, w, _ptr(tmp8), tmp8_dtype, _ptr(rgba0), _ptr(rgba1),
                                        out_dtype, _ptr(y), _stream(stream))


def acnn_frame_refine_out(c, hh, hw, x, dtype, w, bias, y, stream=None) -> int:
    return lib().acnn_frame_refine_out(c, hh, hw, _ptr(x), dtype, _ptr(w), _ptr(bias), _ptr(y),
                                       _stream(stream))


def acnn_film(c, n, dtype, x, t, w0, b0, hn, w2, b2, y, stream=None) -> int:
    return lib().acnn_film(c, n, dtype, _ptr(x), float(t), _ptr(w0), _ptr(b0), hn, _ptr(w2),
                           _ptr(b2), _ptr(y), _stream(stream))


def acnn_last_device_status(stream=None) -> int:
    return lib().acnn_last_device_status(_stream(stream))


def acnn_set_wait_budget(polls: int) -> int:
    return lib().acnn_set_wait_budget(int(polls))


def acnn_section_begin(stream=None) -> int:
    return lib().acnn_section_begin(_stream(stream))


def acnn_section_end(stream=None):
    h = _P()
    st = lib().acnn_section_end(_stream(stream), ctypes.byref(h))
    return st, h.value


def acnn_section_launch(exec_handle, stream=None) -> int:
    return lib().acnn_section_launch(exec_handle, _stream(stream))


def acnn_section_destroy(exec_handle) -> int:
    return lib().acnn_section_destroy(exec_handle)


def acnn_device_sm_count() -> int:
    return lib().acnn_device_sm_count()


# ------------------------------------------------------------------ tensor helpers
def dtype_code(t: torch.dtype) -> int:
    return {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}[t]


def check(status: int, where: str) -> None:
    if status != 0:
        raise AcnnError(status, where)


def conv_desc(x: torch.Tensor, c_out: int, kh: int, kw: int, stride: int, pad: int,
              layout: int) -> ConvDesc:
    if layout == NHWC:
        n, h, w, c = x.shape
    else:
        n, c, h, w = x.shape
    return ConvDesc(n, h, w, c, c_out, kh, kw, stride, pad, layout, dtype_code(x.dtype))


def acnn_conv2d_fused_cat2(desc, x_a, c_a, x_b, w, bias, alpha, residual, res_mode, act, y,
                           workspace, ws_bytes, stream=None) -> int:
    return lib().acnn_conv2d_fused_cat2(ctypes.byref(desc), _ptr(x_a), c_a, _ptr(x_b), _ptr(w),
                                        _ptr(bias), _ptr(alpha), _ptr(residual), res_mode, act,
                                        _ptr(y), _ptr(workspace), ws_bytes, _stream(stream))


def acnn_conv2d_fused_pool2(desc, x, w, bias, alpha, residual, res_mode, act, y, y_pool,
                            stream=None) -> int:
    return lib().acnn_conv2d_fused_pool2(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias),
                                         _ptr(alpha), _ptr(residual), res_mode, act, _ptr(y),
                                         _ptr(y_pool), _stream(stream))


def acnn_conv2d_fused_up2(desc, x_a, c_a, x_b, w, bias, alpha, residual, res_mode, act, y,
                          y_up, workspace, ws_bytes, stream=None) -> int:
    return lib().acnn_conv2d_fused_up2(ctypes.byref(desc), _ptr(x_a), c_a, _ptr(x_b), _ptr(w),
                                       _ptr(bias), _ptr(alpha), _ptr(residual), res_mode, act,
                                       _ptr(y), _ptr(y_up), _ptr(workspace), ws_bytes,
                                       _stream(stream))


def acnn_conv2d_fused_prepacked_staged(desc, x, x_nhwc, w_packed, bias, alpha, residual,
                                       res_mode, act, y, y_nhwc, workspace, ws_bytes,
                                       stream=None) -> int:
    return lib().acnn_conv2d_fused_prepacked_staged(
        ctypes.byref(desc), _ptr(x), _ptr(x_nhwc), _ptr(w_packed), _ptr(bias), _ptr(alpha),
        _ptr(residual), res_mode, act, _ptr(y), _ptr(y_nhwc), _ptr(workspace), ws_bytes,
        _stream(stream))


def acnn_deconv2d_workspace_size(desc, out_dtype) -> int:
    return lib().acnn_deconv2d_workspace_size(ctypes.byref(desc), out_dtype)


def acnn_deconv2d_ws(desc, x, w, bias, alpha, act, out_dtype, y, workspace, ws_bytes,
                     stream=None) -> int:
    return lib().acnn_deconv2d_ws(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias), _ptr(alpha),
                                  act, out_dtype, _ptr(y), _ptr(workspace), ws_bytes,
                                  _stream(stream))


def conv_out_shape(desc: ConvDesc):
    st, oh, ow = acnn_conv2d_out_hw(desc)
    check(st, "acnn_conv2d_out_hw")
    if desc.layout == NHWC:
        return (desc.n, oh, ow, desc.c_out)
    return (desc.n, desc.c_out, oh, ow)


def conv2d_fused(x, w, bias=None, *, stride=1, pad=0, act=ACT_NONE, alpha=None, residual=None,
                 res_mode=RES_NONE, layout=NHWC, out=None, workspace=None, stream=None):
    """y = post(conv(x, w) + bias); w is OHWI for NHWC, OIHW for NCHW."""
    if layout == NHWC:
        c_out, kh, kw, _ = w.shape
    else:
        c_out, _, kh, kw = w.shape
    d = conv_desc(x, c_out, kh, kw, stride, pad, layout)
    y = out if out is not None else torch.empty(conv_out_shape(d), dtype=x.dtype, device=x.device)
    ws_bytes = acnn_conv2d_workspace_size(d)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    st = acnn_conv2d_fused(d, x, w, bias, alpha, residual, res_mode, act, y, workspace,
                           ws_bytes if workspace is not None else 0, stream)
    check(st, "acnn_conv2d_fused")
    return y


def conv2d_fused_pool2(x, w, bias=None, *, act=ACT_NONE, alpha=None, residual=None,
                       res_mode=RES_NONE, out=None, out_pool=None, stream=None):
    """1x1 NHWC conv2d_fused that also returns the 2x2/s2 average pool of its output."""
    c_out = w.shape[0]
    d = conv_desc(x, c_out, 1, 1, 1, 0, NHWC)
    shape = conv_out_shape(d)
    y = out if out is not None else torch.empty(shape, dtype=x.dtype, device=x.device)
    yp = out_pool if out_pool is not None else torch.empty(
        (shape[0], shape[1] // 2, shape[2] // 2, shape[3]), dtype=x.dtype, device=x.device)
    check(acnn_conv2d_fused_pool2(d, x, w, bias, alpha, residual, res_mode, act, y, yp, stream),
          "acnn_conv2d_fused_pool2")
    return y, yp


def conv2d_prepack(desc, w, stream=None):
    """The weights of geometry desc in the form the conv kernels read (a uint8
    device buffer) for conv2d_fused(..., prepacked=True)."""
    wp = torch.empty(acnn_conv2d_prepacked_size(desc), dtype=torch.uint8, device=w.device)
    check(acnn_conv2d_prepack(desc, w, wp, stream), "acnn_conv2d_prepack")
    return wp


def conv2d_fused_cat2(x_a, x_b, w, bias=None, *, stride=1, pad=0, act=ACT_NONE, alpha=None,
                      residual=None, res_mode=RES_NONE, out=None, workspace=None, stream=None):
    """conv2d_fused over torch.cat([x_a, x_b], -1) (NHWC) without building it."""
    n, h, wd, c_a = x_a.shape
    c_b = x_b.shape[3]
    c_out, kh, kw, _ = w.shape
    d = ConvDesc(n, h, wd, c_a + c_b, c_out, kh, kw, stride, pad, NHWC, dtype_code(x_a.dtype))
    y = out if out is not None else torch.empty(conv_out_shape(d), dtype=x_a.dtype,
                                                device=x_a.device)
    ws_bytes = acnn_conv2d_workspace_size(d)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x_a.device)
    st = acnn_conv2d_fused_cat2(d, x_a, c_a, x_b, w, bias, alpha, residual, res_mode, act, y,
                                workspace, ws_bytes if workspace is not None else 0, stream)
    check(st, "acnn_conv2d_fused_cat2")
    return y


def pool2d(x, kind, k, stride, pad, *, layout=NHWC, out=None, stream=None):
    if layout == NHWC:
        n, h, w, c = x.shape
    else:
        n, c, h, w = x.shape
    oh, ow = (h + 2 * pad - k) // stride + 1, (w + 2 * pad - k) // stride + 1
    shape = (n, oh, ow, c) if layout == NHWC else (n, c, oh, ow)
    y = out if out is not None else torch.empty(shape, dtype=x.dtype, device=x.device)
    check(acnn_pool2d(kind, n, h, w, c, k, stride, pad, layout, dtype_code(x.dtype), x, y, stream),
          "acnn_pool2d")
    return y


def resize2d(x, mode, oh, ow, *, layout=NHWC, out_dtype=None, out=None, stream=None):
    if layout == NHWC:
        n, h, w, c = x.shape
    else:
        n, c, h, w = x.shape
    od = out_dtype or x.dtype
    shape = (n, oh, ow, c) if layout == NHWC else (n, c, oh, ow)
    y = out if out is not None else torch.empty(shape, dtype=od, device=x.device)
    check(acnn_resize2d(mode, n, c, h, w, oh, ow, layout, dtype_code(x.dtype), dtype_code(od), x,
                        y, stream), "acnn_resize2d")
    return y


def concat(a, b, *, layout=NHWC, out=None, stream=None):
    if layout == NHWC:
        n, h, w, ca = a.shape
        cb = b.shape[3]
        shape = (n, h, w, ca + cb)
    else:
        n, ca, h, w = a.shape
        cb = b.shape[1]
        shape = (n, ca + cb, h, w)
    y = out if out is not None else torch.empty(shape, dtype=a.dtype, device=a.device)
    check(acnn_concat(n, h, w, ca, cb, layout, dtype_code(a.dtype), a, b, y, stream),
          "acnn_concat")
    return y


def deconv2d(x, w, bias=None, *, act=ACT_NONE, alpha=None, layout=NCHW, out_dtype=None,
             out=None, stream=None):
    """4x4/s2/p1 transposed conv; w is fp32 [CI, CO, 4, 4]."""
    if layout == NHWC:
        n, h, wd, c = x.shape
    else:
        n, c, h, wd = x.shape
    ci, co, kh, kw = w.shape
    d = ConvDesc(n, h, wd, c, co, kh, kw, 2, 1, layout, dtype_code(x.dtype))
    od = out_dtype or x.dtype
    shape = (n, 2 * h, 2 * wd, co) if layout == NHWC else (n, co, 2 * h, 2 * wd)
    y = out if out is not None else torch.empty(shape, dtype=od, device=x.device)
    check(acnn_deconv2d(d, x, w, bias, alpha, act, dtype_code(od), y, stream), "acnn_deconv2d")
    return y


def frame_prep_quarter(rgba0, rgba1, t, *, out_dtype=torch.float16, out=None, stream=None):
    h, w, _ = rgba0.shape
    y = out if out is not None else torch.empty((7, h // 4, w // 4), dtype=out_dtype,
                                                device=rgba0.device)
    check(acnn_frame_prep_quarter(h, w, rgba0, rgba1, t, dtype_code(out_dtype), y, stream),
          "acnn_frame_prep_quarter")
    return y


def frame_flow_out(tmp8, rgba0, rgba1, *, refine_res=None, out=None, stream=None):
    """[5, h/8, w/8] flow/mask map + two h x w RGBA8 frames (+ optional [3, h/4, w/4]
    fp32 refine residual) -> h x w RGBA8 frame."""
    h, w, _ = rgba0.shape
    y = out if out is not None else torch.empty((h, w, 4), dtype=torch.uint8, device=rgba0.device)
    check(acnn_frame_flow_out(h, w, tmp8, dtype_code(tmp8.dtype), rgba0, rgba1, refine_res, y,
                              stream), "acnn_frame_flow_out")
    return y


def frame_refine_prep(tmp8, rgba0, rgba1, *, out_dtype=torch.float16, out=None, stream=None):
    """[5, h/8, w/8] flow/mask map + two frames -> [11, h/4, w/4] refine-head input."""
    h, w, _ = rgba0.shape
    y = out if out is not None else torch.empty((11, h // 4, w // 4), dtype=out_dtype,
                                                device=rgba0.device)
    check(acnn_frame_refine_prep(h, w, tmp8, dtype_code(tmp8.dtype), rgba0, rgba1,
                                 dtype_code(y.dtype), y, stream), "acnn_frame_refine_prep")
    return y


def frame_refine_out(x, w, bias, *, out=None, stream=None):
    """[C, hh, hw] map -> [3, hh, hw] fp32 residual (replicate-padded conv3x3, 2 sigmoid - 1)."""
    c, hh, hw = x.shape
    y = out if out is not None else torch.empty((3, hh, hw), dtype=torch.float32, device=x.device)
    check(acnn_frame_refine_out(c, hh, hw, x, dtype_code(x.dtype), w, bias, y, stream),
          "acnn_frame_refine_out")
    return y


def film(x, t, w0, b0, w2, b2, *, out=None, stream=None):
    """x [C, ...] -> x * (1 + s[c]) + s[C + c], s = the timestep MLP at t."""
    c = x.shape[0]
    n = x.numel() // c
    y = out if out is not None else torch.empty_like(x)
    check(acnn_film(c, n, dtype_code(x.dtype), x, t, w0, b0, b0.numel(), w2, b2, y, stream),
          "acnn_film")
    return y


class Section:
    """One captured CUDA graph: record ABI calls once, replay with launch()."""

    def __init__(self, stream=None):
        self.stream = stream
        self.handle = None

    def __enter__(self):
        check(acnn_section_begin(self.stream), "acnn_section_begin")
        return self

    def __exit__(self, exc_type, exc, tb):
        st, h = acnn_section_end(self.stream)
        if exc_type is None:
            check(st, "acnn_section_end")
        self.handle = h
        return False

    def launch(self, stream=None):
        check(acnn_section_launch(self.handle, stream if stream is not None else self.stream),
              "acnn_section_launch")

    def close(self):
        if self.handle:
            acnn_section_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
