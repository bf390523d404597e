"""Pins for the fp64 oracle: golden closed forms, library routines, invariants.

These tests check the oracle against things other than itself -- closed-form
worked examples under tests/golden/ (each with its citation and derivation),
PyTorch's float64 CPU routines for the special cases that reduce to them,
exact integer arithmetic, and the invariants that the definitions imply -- so
that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails here.  No GPU is used.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


rng = np.random.default_rng(7)


def nhwc_to_nchw(a):
    return np.ascontiguousarray(np.transpose(a, (0, 3, 1, 2)))


def nchw_to_nhwc(a):
    return np.ascontiguousarray(np.transpose(a, (0, 2, 3, 1)))


def ohwi_to_oihw(w):
    return np.ascontiguousarray(np.transpose(w, (0, 3, 1, 2)))


def torch_conv(x_nchw, w_oihw, b, s, p):
    return F.conv2d(torch.from_numpy(x_nchw), torch.from_numpy(w_oihw),
                    None if b is None else torch.from_numpy(np.asarray(b, np.float64)),
                    stride=s, padding=p).numpy()


# --------------------------------------------------------------------------- golden
def test_golden_conv_ones():
    for c in gold("conv_ones_3x3.json")["cases"]:
        x = np.ones((c["N"], c["H"], c["W"], c["C_in"]))
        w = np.ones((c["C_out"], c["K"], c["K"], c["C_in"]))
        y = O.conv2d(x, w, None, stride=c["stride"], pad=c["pad"])
        np.testing.assert_array_equal(y[0, :, :, 0], np.array(c["expected"], float))


def test_golden_maxpool_spike():
    g = gold("maxpool_spike.json")
    x = np.array(g["input"], float)[None, :, :, None]
    y = O.pool2d(x, O.MAX, 3, 2, 1)
    np.testing.assert_array_equal(y[0, :, :, 0], np.array(g["expected"], float))


def test_golden_avgpool():
    g = gold("avgpool_2x2.json")
    x = np.array(g["input"], float)[None, :, :, None]
    y = O.pool2d(x, O.AVG, 2, 2, 0)
    np.testing.assert_array_equal(y[0, :, :, 0], np.array(g["expected"], float))


def test_golden_nearest():
    g = gold("nearest_2x.json")
    x = np.array(g["input"], float)[None, :, :, None]
    y = O.resize2d(x, O.NEAREST, 4, 4)
    np.testing.assert_array_equal(y[0, :, :, 0], np.array(g["expected"], float))


def test_golden_concat():
    g = gold("concat_pixel.json")
    a = np.array(g["a"], float).reshape(1, 1, 1, -1)
    b = np.array(g["b"], float).reshape(1, 1, 1, -1)
    np.testing.assert_array_equal(O.concat(a, b).reshape(-1), np.array(g["expected"], float))


def test_golden_bilinear():
    for c in gold("bilinear.json")["cases"]:
        x = np.array(c["input"], float)[None, None]  # NCHW
        y = O.resize2d(x, O.BILINEAR, c["OH"], c["OW"], layout=O.NCHW)
        np.testing.assert_allclose(y[0, 0], np.array(c["expected"], float), rtol=0, atol=1e-12)


def test_golden_deconv():
    g = gold("deconv_4x4s2p1.json")
    x = np.ones((1, 1, 1, 1))
    w = np.array(g["weight"], float)[None, None]
    y = O.deconv2d(x, w, None)
    np.testing.assert_array_equal(y[0, 0], np.array(g["expected"], float))


def test_golden_prep_quarter():
    g = gold("prep_quarter.json")
    k = np.arange(16).reshape(4, 4)
    f0 = np.zeros((4, 4, 4), np.uint8)
    f0[..., 0] = 17 * k
    f0[..., 1] = 255
    f0[..., 2] = 0
    f0[..., 3] = 99
    f1 = np.zeros((4, 4, 4), np.uint8)
    f1[..., 0] = 0
    f1[..., 1] = 51
    f1[..., 2] = 255 - 17 * k
    y = O.prep_quarter(f0, f1, g["t"])
    np.testing.assert_allclose(y.reshape(-1), np.array(g["expected"]), rtol=0, atol=1e-12)


def test_golden_activations():
    code = {"relu": O.ACT_RELU, "silu": O.ACT_SILU, "prelu": O.ACT_PRELU}
    for name, v, alpha, want in gold("activations.json")["points"]:
        assert O.act(code[name], v, alpha) == pytest.approx(want, abs=1e-15)


def test_golden_round_storage():
    dt = {"bf16": O.BF16, "f16": O.F16}
    for name, v, want in gold("round_storage.json")["cases"]:
        got = O.round_storage([v], dt[name])[0]
        want = math.inf if want == "inf" else want
        assert got == want, (name, v, got, want)


# --------------------------------------------------------------------------- conv
@pytest.mark.parametrize("layout", [O.NHWC, O.NCHW])
@pytest.mark.parametrize("k,s,p", [(3, 1, 1), (3, 2, 1), (1, 1, 0), (1, 2, 0), (4, 2, 1),
                                   (7, 2, 3), (3, 1, 0), (2, 3, 2)])
def test_conv_matches_torch(layout, k, s, p):
    """A plain conv (no act, no residual) is torch's float64 conv2d."""
    n, h, w, cin, cout = 2, 9, 11, 5, 6
    x = rng.standard_normal((n, h, w, cin))
    wt = rng.standard_normal((cout, k, k, cin))
    b = rng.uniform(-0.1, 0.1, cout)
    ref = torch_conv(nhwc_to_nchw(x), ohwi_to_oihw(wt), b, s, p)
    if layout == O.NHWC:
        y = nhwc_to_nchw(O.conv2d(x, wt, b, stride=s, pad=p, layout=O.NHWC))
    else:
        y = O.conv2d(nhwc_to_nchw(x), ohwi_to_oihw(wt), b, stride=s, pad=p, layout=O.NCHW)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_conv_nonsquare_kernel_matches_torch():
    x = rng.standard_normal((1, 7, 8, 3))
    wt = rng.standard_normal((4, 1, 3, 3))  # OHWI, kh=1, kw=3
    ref = torch_conv(nhwc_to_nchw(x), ohwi_to_oihw(wt), None, 1, 0)
    # padding 0 keeps the torch call symmetric-pad compatible
    y = nhwc_to_nchw(O.conv2d(x, wt, None, stride=1, pad=0))
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_conv_1x1_is_matmul():
    x = rng.standard_normal((3, 4, 5, 16))
    wt = rng.standard_normal((8, 1, 1, 16))
    y = O.conv2d(x, wt, None)
    ref = (x.reshape(-1, 16) @ wt.reshape(8, 16).T).reshape(3, 4, 5, 8)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_conv_delta_kernel_identity_and_subsample():
    x = rng.standard_normal((2, 6, 7, 4))
    wt = np.zeros((4, 3, 3, 4))
    for c in range(4):
        wt[c, 1, 1, c] = 1.0
    np.testing.assert_array_equal(O.conv2d(x, wt, None, stride=1, pad=1), x)
    np.testing.assert_array_equal(O.conv2d(x, wt, None, stride=2, pad=1), x[:, ::2, ::2, :])


def _im2col_matmul(x, wt, s, p):
    """Independent second form: explicit patch matrix built by slicing + one matmul."""
    n, h, w, cin = x.shape
    cout, kh, kw, _ = wt.shape
    oh, ow = (h + 2 * p - kh) // s + 1, (w + 2 * p - kw) // s + 1
    xp = np.zeros((n, h + 2 * p, w + 2 * p, cin), x.dtype)
    xp[:, p:p + h, p:p + w, :] = x
    cols = [xp[:, ky:ky + s * (oh - 1) + 1:s, kx:kx + s * (ow - 1) + 1:s, :]
            for ky in range(kh) for kx in range(kw)]
    a = np.concatenate(cols, axis=-1).reshape(n * oh * ow, kh * kw * cin)
    return (a @ wt.reshape(cout, -1).T).reshape(n, oh, ow, cout)


@pytest.mark.parametrize("k,s,p", [(3, 1, 1), (3, 2, 1), (5, 2, 2), (4, 2, 1)])
def test_conv_exact_on_integers(k, s, p):
    """Integer data makes every fp64 partial sum exact: both forms agree bit for bit."""
    x = rng.integers(-3, 4, (2, 9, 10, 6)).astype(np.float64)
    wt = rng.integers(-2, 3, (5, k, k, 6)).astype(np.float64)
    y = O.conv2d(x, wt, None, stride=s, pad=p)
    ref = _im2col_matmul(x.astype(np.int64), wt.astype(np.int64), s, p)
    np.testing.assert_array_equal(y, ref.astype(np.float64))


def test_conv_linearity():
    x1, x2 = rng.standard_normal((2, 1, 6, 6, 3))
    wt = rng.standard_normal((4, 3, 3, 3))
    y = O.conv2d(2.0 * x1 - 3.0 * x2, wt, None, pad=1)
    ref = 2.0 * O.conv2d(x1, wt, None, pad=1) - 3.0 * O.conv2d(x2, wt, None, pad=1)
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("act", [O.ACT_RELU, O.ACT_SILU, O.ACT_PRELU])
@pytest.mark.parametrize("res_mode", [O.RES_NONE, O.RES_ADD_THEN_ACT, O.RES_ACT_THEN_ADD])
def test_conv_epilogue_modes(act, res_mode):
    """Bias, activation and residual compose as the definitions state."""
    x = rng.standard_normal((1, 5, 6, 4))
    wt = rng.standard_normal((3, 3, 3, 4))
    b = rng.uniform(-0.1, 0.1, 3)
    al = rng.uniform(0, 0.25, 3)
    r = rng.standard_normal((1, 5, 6, 3))
    base = nchw_to_nhwc(torch_conv(nhwc_to_nchw(x), ohwi_to_oihw(wt), b, 1, 1))
    tb = torch.from_numpy

    def f(v):
        if act == O.ACT_RELU:
            return F.relu(tb(v)).numpy()
        if act == O.ACT_SILU:
            return F.silu(tb(v)).numpy()
        return F.prelu(tb(nhwc_to_nchw(v)), tb(al)).permute(0, 2, 3, 1).numpy()

    if res_mode == O.RES_NONE:
        ref = f(base)
    elif res_mode == O.RES_ADD_THEN_ACT:
        ref = f(base + r)
    else:
        ref = f(base) + r
    y = O.conv2d(x, wt, b, pad=1, act=act, alpha=al, residual=r, res_mode=res_mode)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_prelu_special_alphas():
    x = rng.standard_normal((1, 4, 4, 3))
    wt = rng.standard_normal((3, 3, 3, 3))
    plain = O.conv2d(x, wt, None, pad=1)
    np.testing.assert_array_equal(
        O.conv2d(x, wt, None, pad=1, act=O.ACT_PRELU, alpha=np.ones(3)), plain)
    np.testing.assert_array_equal(
        O.conv2d(x, wt, None, pad=1, act=O.ACT_PRELU, alpha=np.zeros(3)),
        O.conv2d(x, wt, None, pad=1, act=O.ACT_RELU))


@pytest.mark.parametrize("layout", [O.NHWC, O.NCHW])
def test_conv_points_equal_full(layout):
    x = rng.standard_normal((2, 7, 9, 5))
    wt = rng.standard_normal((6, 3, 3, 5))
    b = rng.uniform(-0.1, 0.1, 6)
    r = rng.standard_normal((2, 4, 5, 6))
    if layout == O.NCHW:
        x, wt, r = nhwc_to_nchw(x), ohwi_to_oihw(wt), nhwc_to_nchw(r)
    full = O.conv2d(x, wt, b, stride=2, pad=1, act=O.ACT_SILU, residual=r,
                    res_mode=O.RES_ACT_THEN_ADD, layout=layout)
    pts = [(0, 0, 0), (1, 3, 4), (1, 2, 1), (0, 3, 0)]
    got = O.conv2d_points(x, wt, b, pts, stride=2, pad=1, act=O.ACT_SILU, residual=r,
                          res_mode=O.RES_ACT_THEN_ADD, layout=layout)
    for i, (n, oy, ox) in enumerate(pts):
        ref = full[n, oy, ox, :] if layout == O.NHWC else full[n, :, oy, ox]
        np.testing.assert_array_equal(got[i], ref)


def test_conv_threading_is_deterministic():
    x = rng.standard_normal((2, 8, 8, 7))
    wt = rng.standard_normal((5, 3, 3, 7))
    a = O.conv2d(x, wt, None, pad=1, threads=1)
    b = O.conv2d(x, wt, None, pad=1, threads=5)
    np.testing.assert_array_equal(a, b)


# --------------------------------------------------------------------------- pools
@pytest.mark.parametrize("layout", [O.NHWC, O.NCHW])
@pytest.mark.parametrize("hw", [(8, 8), (7, 9), (1, 1), (2, 5)])
def test_maxpool_matches_torch(layout, hw):
    x = rng.standard_normal((2, 3) + hw)  # NCHW
    ref = F.max_pool2d(torch.from_numpy(x), 3, 2, 1).numpy()
    if layout == O.NHWC:
        y = nhwc_to_nchw(O.pool2d(nchw_to_nhwc(x), O.MAX, 3, 2, 1))
    else:
        y = O.pool2d(x, O.MAX, 3, 2, 1, layout=O.NCHW)
    np.testing.assert_array_equal(y, ref)


def test_maxpool_constant_map():
    x = np.full((1, 6, 5, 2), -7.25)
    np.testing.assert_array_equal(O.pool2d(x, O.MAX, 3, 2, 1), np.full((1, 3, 3, 2), -7.25))


@pytest.mark.parametrize("layout", [O.NHWC, O.NCHW])
def test_avgpool_matches_torch_and_inverts_nearest(layout):
    x = rng.standard_normal((2, 4, 6, 8))  # NCHW
    ref = F.avg_pool2d(torch.from_numpy(x), 2, 2).numpy()
    if layout == O.NHWC:
        y = nhwc_to_nchw(O.pool2d(nchw_to_nhwc(x), O.AVG, 2, 2, 0))
        up = O.resize2d(nchw_to_nhwc(x), O.NEAREST, 12, 16)
        back = nhwc_to_nchw(O.pool2d(up, O.AVG, 2, 2, 0))
    else:
        y = O.pool2d(x, O.AVG, 2, 2, 0, layout=O.NCHW)
        up = O.resize2d(x, O.NEAREST, 12, 16, layout=O.NCHW)
        back = O.pool2d(up, O.AVG, 2, 2, 0, layout=O.NCHW)
    np.testing.assert_allclose(y, ref, rtol=1e-14, atol=1e-15)
    np.testing.assert_array_equal(back, x)


def test_avgpool_constant_and_depthwise_conv():
    x = np.full((1, 4, 4, 3), 2.5)
    np.testing.assert_array_equal(O.pool2d(x, O.AVG, 2, 2, 0), np.full((1, 2, 2, 3), 2.5))
    x = rng.standard_normal((1, 6, 4, 3))
    wt = np.zeros((3, 2, 2, 3))
    for c in range(3):
        wt[c, :, :, c] = 0.25
    np.testing.assert_allclose(O.pool2d(x, O.AVG, 2, 2, 0), O.conv2d(x, wt, None, stride=2),
                               rtol=1e-14, atol=1e-15)


# --------------------------------------------------------------------------- resize
@pytest.mark.parametrize("layout", [O.NHWC, O.NCHW])
def test_nearest_2x_matches_torch(layout):
    x = rng.standard_normal((2, 3, 5, 4))
    ref = F.interpolate(torch.from_numpy(x), scale_factor=2, mode="nearest").numpy()
    if layout == O.NHWC:
        y = nhwc_to_nchw(O.resize2d(nchw_to_nhwc(x), O.NEAREST, 10, 8))
    else:
        y = O.resize2d(x, O.NEAREST, 10, 8, layout=O.NCHW)
    np.testing.assert_array_equal(y, ref)


@pytest.mark.parametrize("layout", [O.NHWC, O.NCHW])
@pytest.mark.parametrize("io", [((16, 24), (4, 6)), ((5, 7), (40, 56)), ((9, 13), (4, 17)),
                                ((1, 1), (3, 2)), ((6, 6), (6, 6))])
def test_bilinear_matches_torch(layout, io):
    (h, w), (oh, ow) = io
    x = rng.standard_normal((2, 3, h, w))
    ref = F.interpolate(torch.from_numpy(x), size=(oh, ow), mode="bilinear",
                        align_corners=False).numpy()
    if layout == O.NHWC:
        y = nhwc_to_nchw(O.resize2d(nchw_to_nhwc(x), O.BILINEAR, oh, ow))
    else:
        y = O.resize2d(x, O.BILINEAR, oh, ow, layout=O.NCHW)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_bilinear_invariants():
    c = np.full((1, 1, 7, 9), 3.5)
    np.testing.assert_allclose(O.resize2d(c, O.BILINEAR, 21, 4, layout=O.NCHW), 3.5,
                               rtol=0, atol=1e-14)
    x = rng.standard_normal((1, 2, 5, 6))
    np.testing.assert_array_equal(O.resize2d(x, O.BILINEAR, 5, 6, layout=O.NCHW), x)
    # a linear ramp along x is reproduced wherever both taps are in range
    ramp = np.tile(np.arange(16, dtype=float), (1, 1, 3, 1))
    y = O.resize2d(ramp, O.BILINEAR, 3, 64, layout=O.NCHW)
    src = (np.arange(64) + 0.5) * (16 / 64) - 0.5
    inside = (src >= 0) & (src <= 15)
    np.testing.assert_allclose(y[0, 0, 1, inside], src[inside], rtol=0, atol=1e-12)
    # 1/4 downsample is the mean of the centre 2x2 of each 4x4 block (src = 4*dst + 1.5)
    x = rng.standard_normal((1, 1, 8, 12))
    q = O.resize2d(x, O.BILINEAR, 2, 3, layout=O.NCHW)
    blocks = x[0, 0].reshape(2, 4, 3, 4)[:, 1:3, :, 1:3].mean(axis=(1, 3))
    np.testing.assert_allclose(q[0, 0], blocks, rtol=0, atol=1e-14)


# --------------------------------------------------------------------------- concat
@pytest.mark.parametrize("layout", [O.NHWC, O.NCHW])
def test_concat_slices_back(layout):
    a = rng.standard_normal((2, 3, 4, 5))
    b = rng.standard_normal((2, 3, 4, 7))
    if layout == O.NCHW:
        a = rng.standard_normal((2, 5, 3, 4))
        b = rng.standard_normal((2, 7, 3, 4))
        y = O.concat(a, b, layout=O.NCHW)
        np.testing.assert_array_equal(y[:, :5], a)
        np.testing.assert_array_equal(y[:, 5:], b)
    else:
        y = O.concat(a, b)
        np.testing.assert_array_equal(y[..., :5], a)
        np.testing.assert_array_equal(y[..., 5:], b)


# --------------------------------------------------------------------------- deconv
@pytest.mark.parametrize("layout", [O.NCHW, O.NHWC])
@pytest.mark.parametrize("k,s,p", [(4, 2, 1), (3, 2, 1), (2, 2, 0)])
def test_deconv_matches_torch(layout, k, s, p):
    x = rng.standard_normal((2, 6, 5, 7))  # NCHW
    w = rng.standard_normal((6, 3, k, k))
    b = rng.uniform(-0.1, 0.1, 3)
    ref = F.conv_transpose2d(torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(b),
                             stride=s, padding=p).numpy()
    if layout == O.NCHW:
        y = O.deconv2d(x, w, b, k=k, s=s, p=p)
    else:
        y = nhwc_to_nchw(O.deconv2d(nchw_to_nhwc(x), w, b, k=k, s=s, p=p, layout=O.NHWC))
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_deconv_adjoint_of_conv():
    """<deconv_w(x), y> = <x, conv_w(y)> with the conv 4x4/s2/p1 sharing w."""
    x = rng.standard_normal((1, 4, 5, 6))      # NCHW, CI = 4 (the deconv input)
    w = rng.standard_normal((4, 3, 4, 4))      # [CI, CO, K, K]
    yv = rng.standard_normal((1, 3, 10, 12))   # deconv output shape
    d = O.deconv2d(x, w, None)
    # conv from CO=3 channels back to CI=4 channels: OIHW weight = w as [CI, CO, K, K]
    c = O.conv2d(yv, w, None, stride=2, pad=1, layout=O.NCHW)
    np.testing.assert_allclose(np.sum(d * yv), np.sum(x * c), rtol=1e-11)


def test_deconv_zero_insertion_form():
    """Deconv = zero-insertion upsample then conv with the flipped kernel, pad K-1-P."""
    x = rng.standard_normal((1, 3, 4, 5))
    w = rng.standard_normal((3, 2, 4, 4))
    z = np.zeros((1, 3, 7, 9))
    z[:, :, ::2, ::2] = x
    wf = np.ascontiguousarray(np.transpose(w[:, :, ::-1, ::-1], (1, 0, 2, 3)))
    ref = O.conv2d(z, wf, None, stride=1, pad=2, layout=O.NCHW)
    # the zero-inserted map is one short of 2*IH; the last row/col of taps is all padding
    y = O.deconv2d(x, w, None)
    np.testing.assert_allclose(y[:, :, :ref.shape[2], :ref.shape[3]], ref, rtol=1e-12,
                               atol=1e-12)


# --------------------------------------------------------------------------- prep + rounding
def test_prep_quarter_matches_torch():
    h, w = 16, 24
    f0 = rng.integers(0, 256, (h, w, 4)).astype(np.uint8)
    f1 = rng.integers(0, 256, (h, w, 4)).astype(np.uint8)
    y = O.prep_quarter(f0, f1, 0.5)
    planes = np.stack([f0[..., 2], f0[..., 1], f0[..., 0], f1[..., 2], f1[..., 1], f1[..., 0]])
    ref = F.interpolate(torch.from_numpy(planes[None].astype(np.float64) / 255.0),
                        size=(h // 4, w // 4), mode="bilinear", align_corners=False).numpy()[0]
    np.testing.assert_allclose(y[:6], ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(y[6], 0.5)


@pytest.mark.parametrize("dt,tdt", [(O.BF16, torch.bfloat16), (O.F16, torch.float16),
                                    (O.F32, torch.float32)])
def test_round_storage_matches_torch_cast(dt, tdt):
    """On values exactly representable in fp32, RNE to the narrow type is torch's cast."""
    v = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 6, 20000),
        np.ldexp(rng.integers(1, 2 ** 12, 4000), rng.integers(-40, 0, 4000)).astype(float),
        [0.0, -0.0, 65504.0, 65519.0, 65520.0, -65536.0, 1e-40, 3.0e38],
    ]).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(v.astype(np.float32)).to(tdt).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_storage(v, dt), ref)


# --------------------------------------------------------------------------- flow out (NEXT-1)
# P3 "@framecast/rt 1.0.0 -- package/rt.js", wgslFlowOut: x8 bilinear upsample of
# the flow/mask map, backward warp of both frames, sigmoid-mask blend, truncating
# RGBA8 pack, all in binary32.  The pins below restate the page's arithmetic in
# numpy float32 (one operation at a time, so nothing is fused) for inputs where
# the warp or the blend reduce to a closed form.
f32 = np.float32


def _unit(bytes_):
    return bytes_.astype(f32) / f32(255)


def _byte(v):
    return np.floor(np.clip(v, f32(0), f32(1)) * f32(255)).astype(np.uint8)


def _flow_map(h, w, u0=0.0, v0=0.0, u1=0.0, v1=0.0, mask=0.0):
    """Constant planes: flow values are in 1/8-resolution units (x8 on the page)."""
    t = np.empty((5, h // 8, w // 8), f32)
    for c, val in enumerate((u0, v0, u1, v1, mask)):
        t[c] = val
    return t


def _frames(h, w, seed=5):
    g = np.random.default_rng(seed)
    return (g.integers(0, 256, (h, w, 4)).astype(np.uint8),
            g.integers(0, 256, (h, w, 4)).astype(np.uint8))


@pytest.mark.parametrize("mask,which", [(30.0, 0), (-30.0, 1)])
def test_flow_out_identity_picks_one_frame(mask, which):
    """Zero flow and a saturated mask: the output is one frame's bytes after the
    page's byte -> /255 -> *255 -> truncation round trip; alpha 255."""
    h, w = 24, 40
    f0, f1 = _frames(h, w)
    out = O.flow_out(_flow_map(h, w, mask=mask), f0, f1)
    src = (f0, f1)[which]
    np.testing.assert_array_equal(out[..., :3], _byte(_unit(src[..., :3])))
    assert (out[..., 3] == 255).all()


@pytest.mark.parametrize("shift", [1, 2, -3, 17])
def test_flow_out_integer_shift_is_clamped_translation(shift):
    """flow0.x = shift pixels (shift/8 at 1/8 resolution): out(x) = frame0(clamp(x + shift))."""
    h, w = 16, 48
    f0, f1 = _frames(h, w, seed=7)
    out = O.flow_out(_flow_map(h, w, u0=shift / 8.0, mask=30.0), f0, f1)
    xs = np.clip(np.arange(w) + shift, 0, w - 1)
    np.testing.assert_array_equal(out[..., :3], _byte(_unit(f0[:, xs, :3])))


def test_flow_out_half_pixel_shift_is_bilinear_mean():
    """flow1.y = +0.5 px: out(y) = mix(frame1(y), frame1(y+1), 0.5) with mix(a,b,f) = a(1-f)+bf."""
    h, w = 24, 16
    f0, f1 = _frames(h, w, seed=9)
    out = O.flow_out(_flow_map(h, w, v1=0.5 / 8.0, mask=-30.0), f0, f1)
    a = _unit(f1[:, :, :3])
    b = _unit(f1[np.clip(np.arange(h) + 1, 0, h - 1), :, :3])
    ref = a * f32(0.5) + b * f32(0.5)
    np.testing.assert_array_equal(out[..., :3], _byte(ref))


@pytest.mark.parametrize("ca,cb", [(0, 255), (100, 37), (255, 254), (1, 2)])
def test_flow_out_mask_zero_blends_halves(ca, cb):
    """Mask logit 0: m = 1/(1+e^0) = 0.5 exactly; constant frames give a constant
    v = (ca/255)*0.5 + (cb/255)*0.5 in every channel."""
    h, w = 16, 16
    f0 = np.full((h, w, 4), ca, np.uint8)
    f1 = np.full((h, w, 4), cb, np.uint8)
    out = O.flow_out(_flow_map(h, w, u0=0.3, v1=-0.7, mask=0.0), f0, f1)
    v = f32(ca) / f32(255) * f32(0.5) + f32(cb) / f32(255) * f32(0.5)
    assert (out[..., :3] == _byte(np.array([v], f32))[0]).all()


def test_flow_out_sigmoid_and_upsample_positions():
    """Frame 0 all 255, frame 1 all 0: the clamped pre-byte value is the mask
    m = 1/(1+exp(-l)) of the x8-upsampled logit l.  With a logit plane that is
    linear in x at 1/8 resolution, l at output x is the line at the align_corners=
    false source position (x + 0.5)/8 - 0.5, clamped to the plane; m matches
    float64 arithmetic to a few float32 ulps (the page's exp is binary32)."""
    h, w = 8, 64
    f0 = np.full((h, w, 4), 255, np.uint8)
    f1 = np.zeros((h, w, 4), np.uint8)
    t = _flow_map(h, w)
    t[4] = (np.arange(w // 8, dtype=f32) * f32(2.0) - f32(7.0))[None, :]  # -7, -5, ..., 7
    out, pre = O.flow_out(t, f0, f1, with_pre=True)
    sx = (np.arange(w) + 0.5) / 8.0 - 0.5
    l = np.clip(sx, 0, w // 8 - 1) * 2.0 - 7.0
    m = 1.0 / (1.0 + np.exp(-l))
    for c in range(3):
        np.testing.assert_allclose(pre[c], np.broadcast_to(m, (h, w)), rtol=4e-7, atol=0)


def test_flow_out_exp_wide_range():
    """The binary32 exp inside the mask stays within 2 ulp of float64 over
    [-80, 80] (pinned through the sigmoid of constant-frame blends)."""
    h, w = 8, 8
    f0 = np.full((h, w, 4), 255, np.uint8)
    f1 = np.zeros((h, w, 4), np.uint8)
    for l in np.linspace(-80.0, 80.0, 161).astype(f32):
        _, pre = O.flow_out(_flow_map(h, w, mask=float(l)), f0, f1, with_pre=True)
        ref = 1.0 / (1.0 + math.exp(-float(l)))
        assert abs(float(pre[0, 0, 0]) - ref) <= 3 * np.spacing(f32(ref)) + 1e-45, (l, pre[0, 0, 0], ref)


def test_flow_out_far_flow_clamps_to_border():
    """A flow far outside the frame samples the clamped border pixel."""
    h, w = 16, 16
    f0, f1 = _frames(h, w, seed=11)
    out = O.flow_out(_flow_map(h, w, u0=1e6, v0=-1e6, mask=30.0), f0, f1)
    corner = _byte(_unit(f0[0, w - 1, :3]))
    assert (out[..., :3] == corner).all()


# --------------------------------------------------------------------------- t-factored stack (NEXT-3)
# P3 "@framecast/rt 1.0.0 -- package/rt.js": wgslFilm + filmParams (FiLM of the
# trunk features by a per-timestep MLP), wgslRefinePrep, wgslRefineOut, and the
# refine residual folded into the flow-out stage.
def test_film_matches_torch_mlp():
    """s = Linear2(relu(Linear1(t))) is torch's linear + relu; FiLM is x*(1+s_c)+s_{C+c}."""
    c, hn = 6, 5
    x = rng.standard_normal((c, 4, 7))
    w0, b0 = rng.standard_normal(hn), rng.standard_normal(hn)
    w2, b2 = rng.standard_normal((2 * c, hn)), rng.standard_normal(2 * c)
    t = 0.37
    h = F.relu(F.linear(torch.tensor([[t]], dtype=torch.float64), torch.from_numpy(w0[:, None]),
                        torch.from_numpy(b0)))
    s = F.linear(h, torch.from_numpy(w2), torch.from_numpy(b2))[0].numpy()
    ref = x * (1.0 + s[:c, None, None]) + s[c:, None, None]
    np.testing.assert_allclose(O.film(x, t, w0, b0, w2, b2), ref, rtol=1e-12, atol=1e-12)


def test_film_dead_hidden_units_and_identity():
    """All hidden units negative (relu = 0): s = b2; b2 = 0 then gives the identity."""
    c = 3
    x = rng.standard_normal((c, 10))
    w0, b0 = np.ones(4), -np.ones(4) * 5.0  # w0 t + b0 < 0 for t < 5
    w2 = rng.standard_normal((2 * c, 4))
    np.testing.assert_array_equal(O.film(x, 1.0, w0, b0, w2, np.zeros(2 * c)), x)
    b2 = np.array([0.5, -1.0, 0.0, 2.0, 0.25, -3.0])
    np.testing.assert_allclose(O.film(x, 1.0, w0, b0, w2, b2),
                               x * (1 + b2[:c, None]) + b2[c:, None], rtol=1e-15, atol=0)


def test_refine_prep_zero_flow_is_quarter_bilinear():
    """With zero flow the warped planes are the frames, and the mean over the centre
    2x2 of each 4x4 block is torch's bilinear 1/4 resize (align_corners=False)."""
    h, w = 16, 24
    f0, f1 = _frames(h, w, seed=13)
    t = np.zeros((5, h // 8, w // 8))
    t[4] = 0.7
    y = O.refine_prep(t, f0, f1)
    for f, off in ((f0, 0), (f1, 3)):
        planes = np.stack([f[..., 2], f[..., 1], f[..., 0]]).astype(np.float64) / 255.0
        ref = F.interpolate(torch.from_numpy(planes[None]), size=(h // 4, w // 4),
                            mode="bilinear", align_corners=False).numpy()[0]
        np.testing.assert_allclose(y[off:off + 3], ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y[6], 1.0 / (1.0 + math.exp(-0.7)), rtol=1e-14)
    np.testing.assert_array_equal(y[7:], 0.0)


def test_refine_prep_constant_flow_channels():
    """A constant flow value u at 1/8 resolution is 8u pixels; the flow planes hold
    the mean flow times 0.25/20 = u/10."""
    h, w = 16, 16
    f0, f1 = _frames(h, w, seed=15)
    t = np.zeros((5, h // 8, w // 8))
    t[0], t[1], t[2], t[3] = 0.5, -0.25, 1.5, 0.125
    y = O.refine_prep(t, f0, f1)
    for k, u in enumerate((0.5, -0.25, 1.5, 0.125)):
        np.testing.assert_allclose(y[7 + k], u / 10.0, rtol=1e-14)


def test_refine_out_is_replicate_padded_conv_then_2sigmoid_minus_1():
    c, hh, hw = 5, 7, 9
    x = rng.standard_normal((c, hh, hw))
    w = rng.standard_normal((3, c, 3, 3))
    b = rng.standard_normal(3)
    xp = F.pad(torch.from_numpy(x[None]), (1, 1, 1, 1), mode="replicate")
    acc = F.conv2d(xp, torch.from_numpy(w), torch.from_numpy(b)).numpy()[0]
    np.testing.assert_allclose(O.refine_out(x, w, b), 2.0 / (1.0 + np.exp(-acc)) - 1.0,
                               rtol=1e-12, atol=1e-12)


def test_flow_out_constant_refine_residual_is_added_before_clamp():
    """Identity warp (mask saturated to frame 0) plus a constant residual r per channel
    (exact in binary32, so its x4 upsample is r): byte = trunc(clamp(p + r) * 255)."""
    h, w = 16, 24
    f0, f1 = _frames(h, w, seed=17)
    res = np.empty((3, h // 4, w // 4), f32)
    res[0], res[1], res[2] = 0.125, -0.25, 0.5  # B, G, R
    out = O.flow_out(_flow_map(h, w, mask=30.0), f0, f1, res=res)
    for k, (byte, r) in enumerate(((2, 0.125), (1, -0.25), (0, 0.5))):
        ref = _byte(_unit(f0[..., byte]) + f32(r))
        np.testing.assert_array_equal(out[..., byte], ref, err_msg=f"channel {k}")
