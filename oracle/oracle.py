"""Python face of the fp64 CPU oracle (``acnn_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this module; the product library
never does.  It shares no code with the CUDA path.  Arrays are numpy float64
in the same layouts as the GPU tensors (NHWC or NCHW activations; OHWI or
OIHW conv weights; [CI, CO, K, K] deconv weights).

``build()`` compiles the C file with gcc (no BLAS, no SIMD intrinsics,
plain ``-O2``) into ``liboracle.so`` beside it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "acnn_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

NHWC, NCHW = 0, 1
ACT_NONE, ACT_RELU, ACT_SILU, ACT_PRELU = 0, 1, 2, 3
RES_NONE, RES_ADD_THEN_ACT, RES_ACT_THEN_ADD = 0, 1, 2
F32, F16, BF16 = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared",
           "-ffp-contract=off", SRC, "-o", tmp, "-lm", "-lpthread"]
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


def nthreads() -> int:
    """Host threads the oracle uses: the cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(LIB)
    d = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.oracle_conv2d.argtypes = [i] * 10 + [d] * 5 + [i, i, d, i]
    lib.oracle_conv2d_points.argtypes = ([i] * 10 + [d] * 5 + [i, i,
                                         ctypes.POINTER(ctypes.c_int), i, d, i])
    lib.oracle_pool2d.argtypes = [i] * 9 + [d, d, i]
    lib.oracle_resize2d.argtypes = [i] * 8 + [d, d, i]
    lib.oracle_concat.argtypes = [i] * 6 + [d, d, d]
    lib.oracle_deconv2d.argtypes = [i] * 9 + [d] * 4 + [i, d, i]
    lib.oracle_prep_quarter.argtypes = [i, i, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_double, d]
    lib.oracle_flow_out.argtypes = [i, i, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, i]
    lib.oracle_film.argtypes = [i, i, d, ctypes.c_double, d, d, i, d, d, d]
    lib.oracle_refine_prep.argtypes = [i, i, d, ctypes.c_void_p, ctypes.c_void_p, d]
    lib.oracle_refine_out.argtypes = [i, i, i, d, d, d, d]
    lib.oracle_round_storage.argtypes = [d, ctypes.c_size_t, i]
    lib.oracle_round_value.argtypes = [ctypes.c_double, i]
    lib.oracle_round_value.restype = ctypes.c_double
    lib.oracle_act.argtypes = [i, ctypes.c_double, ctypes.c_double]
    lib.oracle_act.restype = ctypes.c_double
    lib.oracle_conv_out.argtypes = [i, i, i, i]
    for f in ("oracle_conv2d", "oracle_conv2d_points", "oracle_pool2d", "oracle_resize2d",
              "oracle_concat", "oracle_deconv2d", "oracle_prep_quarter", "oracle_conv_out"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def conv_out(size: int, k: int, s: int, p: int) -> int:
    return (size + 2 * p - k) // s + 1


def _geom(x, layout):
    if layout == NHWC:
        n, h, w, c = x.shape
    else:
        n, c, h, w = x.shape
    return n, c, h, w


def _shape(layout, n, c, h, w):
    return (n, h, w, c) if layout == NHWC else (n, c, h, w)


def conv2d(x, w, bias=None, *, stride=1, pad=0, act=ACT_NONE, alpha=None,
           residual=None, res_mode=RES_NONE, layout=NHWC, threads=None):
    """fp64 conv2d_fused.  x NHWC/NCHW, w OHWI (NHWC) or OIHW (NCHW)."""
    lib = _load()
    x, w, bias, alpha, residual = map(_f64, (x, w, bias, alpha, residual))
    n, cin, h, wd = _geom(x, layout)
    if layout == NHWC:
        cout, kh, kw, cin_w = w.shape
    else:
        cout, cin_w, kh, kw = w.shape
    assert cin_w == cin, (cin_w, cin)
    oh, ow = conv_out(h, kh, stride, pad), conv_out(wd, kw, stride, pad)
    y = np.empty(_shape(layout, n, cout, oh, ow), np.float64)
    rc = lib.oracle_conv2d(layout, n, h, wd, cin, cout, kh, kw, stride, pad,
                           _ptr(x), _ptr(w), _ptr(bias), _ptr(alpha), _ptr(residual),
                           res_mode, act, _ptr(y), threads or nthreads())
    assert rc == 0
    return y


def conv2d_points(x, w, bias, pts, *, stride=1, pad=0, act=ACT_NONE, alpha=None,
                  residual=None, res_mode=RES_NONE, layout=NHWC, threads=None):
    """fp64 conv2d_fused at output pixels pts[i] = (n, oy, ox); returns [npts, C_out]."""
    lib = _load()
    x, w, bias, alpha, residual = map(_f64, (x, w, bias, alpha, residual))
    n, cin, h, wd = _geom(x, layout)
    if layout == NHWC:
        cout, kh, kw, _ = w.shape
    else:
        cout, _, kh, kw = w.shape
    pts = np.ascontiguousarray(np.asarray(pts, dtype=np.int32).reshape(-1, 3))
    y = np.empty((pts.shape[0], cout), np.float64)
    rc = lib.oracle_conv2d_points(layout, n, h, wd, cin, cout, kh, kw, stride, pad,
                                  _ptr(x), _ptr(w), _ptr(bias), _ptr(alpha), _ptr(residual),
                                  res_mode, act,
                                  pts.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                  pts.shape[0], _ptr(y), threads or nthreads())
    assert rc == 0
    return y


MAX, AVG = 0, 1


def pool2d(x, kind, k, s, p, *, layout=NHWC, threads=None):
    lib = _load()
    x = _f64(x)
    n, c, h, w = _geom(x, layout)
    oh, ow = conv_out(h, k, s, p), conv_out(w, k, s, p)
    y = np.empty(_shape(layout, n, c, oh, ow), np.float64)
    rc = lib.oracle_pool2d(kind, layout, n, c, h, w, k, s, p, _ptr(x), _ptr(y),
                           threads or nthreads())
    assert rc == 0
    return y


NEAREST, BILINEAR = 0, 1


def resize2d(x, mode, oh, ow, *, layout=NHWC, threads=None):
    lib = _load()
    x = _f64(x)
    n, c, h, w = _geom(x, layout)
    y = np.empty(_shape(layout, n, c, oh, ow), np.float64)
    rc = lib.oracle_resize2d(mode, layout, n, c, h, w, oh, ow, _ptr(x), _ptr(y),
                             threads or nthreads())
    assert rc == 0
    return y


def concat(a, b, *, layout=NHWC):
    lib = _load()
    a, b = _f64(a), _f64(b)
    n, ca, h, w = _geom(a, layout)
    _, cb, _, _ = _geom(b, layout)
    y = np.empty(_shape(layout, n, ca + cb, h, w), np.float64)
    rc = lib.oracle_concat(layout, n, h, w, ca, cb, _ptr(a), _ptr(b), _ptr(y))
    assert rc == 0
    return y


def deconv2d(x, w, bias=None, *, k=4, s=2, p=1, act=ACT_NONE, alpha=None, layout=NCHW,
             threads=None):
    """fp64 transposed conv, weight [CI, CO, K, K] (P3 wgslDeconv)."""
    lib = _load()
    x, w, bias, alpha = map(_f64, (x, w, bias, alpha))
    n, cin, h, wd = _geom(x, layout)
    cin_w, cout, kh, kw = w.shape
    assert cin_w == cin and kh == k and kw == k
    oh, ow = (h - 1) * s - 2 * p + k, (wd - 1) * s - 2 * p + k
    y = np.empty(_shape(layout, n, cout, oh, ow), np.float64)
    rc = lib.oracle_deconv2d(layout, n, h, wd, cin, cout, k, s, p, _ptr(x), _ptr(w),
                             _ptr(bias), _ptr(alpha), act, _ptr(y), threads or nthreads())
    assert rc == 0
    return y


def prep_quarter(rgba0, rgba1, t):
    """Two [H, W, 4] uint8 RGBA frames -> [7, H/4, W/4] fp64 (P3 wgslPrepQuarter)."""
    lib = _load()
    a = np.ascontiguousarray(rgba0, dtype=np.uint8)
    b = np.ascontiguousarray(rgba1, dtype=np.uint8)
    h, w, four = a.shape
    assert four == 4 and b.shape == a.shape
    y = np.empty((7, h // 4, w // 4), np.float64)
    rc = lib.oracle_prep_quarter(h, w, a.ctypes.data, b.ctypes.data, float(t), _ptr(y))
    assert rc == 0
    return y


def flow_out(tmp8, rgba0, rgba1, *, res=None, with_pre=False, threads=None):
    """P3 wgslFlowOut: [5, H/8, W/8] flow/mask (float32) + two [H, W, 4] uint8
    frames -> [H, W, 4] uint8 (and, with_pre, the clamped R, G, B [3, H, W]
    float32 before the byte scale).  res: the t-factored stack's refine
    residual [3, H/4, W/4] (B, G, R, float32), upsampled x4 and added before
    the clamp.  Computed in binary32, as on the page."""
    lib = _load()
    a = np.ascontiguousarray(rgba0, dtype=np.uint8)
    b = np.ascontiguousarray(rgba1, dtype=np.uint8)
    h, w, four = a.shape
    assert four == 4 and b.shape == a.shape and h % 8 == 0 and w % 8 == 0
    t = np.ascontiguousarray(tmp8, dtype=np.float32)
    assert t.shape == (5, h // 8, w // 8)
    out = np.empty((h, w, 4), np.uint8)
    pre = np.empty((3, h, w), np.float32) if with_pre else None
    r = None
    if res is not None:
        r = np.ascontiguousarray(res, dtype=np.float32)
        assert r.shape == (3, h // 4, w // 4)
    rc = lib.oracle_flow_out(h, w, t.ctypes.data, a.ctypes.data, b.ctypes.data,
                             r.ctypes.data if r is not None else None, out.ctypes.data,
                             pre.ctypes.data if with_pre else None, threads or nthreads())
    assert rc == 0
    return (out, pre) if with_pre else out


def film(x, t, w0, b0, w2, b2):
    """P3 wgslFilm with filmParams: x [C, N] (any trailing shape) -> x * (1 + s[c])
    + s[C + c], s = b2 + W2 relu(w0 t + b0) (W2 [2C, HN])."""
    lib = _load()
    x = _f64(x)
    c = x.shape[0]
    n = x.size // c
    w0, b0, w2, b2 = _f64(w0).ravel(), _f64(b0).ravel(), _f64(w2), _f64(b2).ravel()
    hn = w0.size
    assert w2.shape == (2 * c, hn) and b2.size == 2 * c
    y = np.empty_like(x)
    assert lib.oracle_film(c, n, _ptr(x), float(t), _ptr(w0), _ptr(b0), hn, _ptr(w2), _ptr(b2),
                           _ptr(y)) == 0
    return y


def refine_prep(tmp8, rgba0, rgba1):
    """P3 wgslRefinePrep: [5, H/8, W/8] + two [H, W, 4] frames -> [11, H/4, W/4]."""
    lib = _load()
    a = np.ascontiguousarray(rgba0, dtype=np.uint8)
    b = np.ascontiguousarray(rgba1, dtype=np.uint8)
    h, w, _ = a.shape
    t = _f64(tmp8)
    assert t.shape == (5, h // 8, w // 8)
    y = np.empty((11, h // 4, w // 4), np.float64)
    assert lib.oracle_refine_prep(h, w, _ptr(t), a.ctypes.data, b.ctypes.data, _ptr(y)) == 0
    return y


def refine_out(x, w, b):
    """P3 wgslRefineOut: x [C, HH, HW], w [3, C, 3, 3], b [3] -> 2 sigmoid(conv) - 1
    with replicate padding, [3, HH, HW]."""
    lib = _load()
    x, w, b = _f64(x), _f64(w), _f64(b).ravel()
    c, hh, hw = x.shape
    assert w.shape == (3, c, 3, 3)
    y = np.empty((3, hh, hw), np.float64)
    assert lib.oracle_refine_out(c, hh, hw, _ptr(x), _ptr(w), _ptr(b), _ptr(y)) == 0
    return y


def round_storage(v, dtype):
    """Round every value to the storage type (F32/F16/BF16), ties to even."""
    lib = _load()
    v = np.array(v, dtype=np.float64, copy=True, order="C")
    lib.oracle_round_storage(_ptr(v), v.size, dtype)
    return v


def act(code, v, alpha=0.0):
    return _load().oracle_act(code, float(v), float(alpha))


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
