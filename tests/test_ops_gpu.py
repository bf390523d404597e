"""Parity of every ABI op (CUDA, through the C ABI) with the fp64 oracle.

Sizes span several tiles with ragged tails; inputs are the seeded generators
of activation_cnn_gb300.inputs.  Max-pool, nearest resize and concat must be
bit-exact; integer-valued conv cases must be bit-exact too (every fp32 partial
sum is exact, so the one rounding at the store is the oracle's rounding).
"""
import numpy as np
import pytest
import torch

from activation_cnn_gb300 import acnn as A
from activation_cnn_gb300 import inputs as G
from oracle import oracle as O
from tests.parity import (Guarded, assert_bitexact, assert_bytes_boundary, assert_parity,
                           guarded_bytes, to64)

pytestmark = pytest.mark.gpu

DT = {"f32": G.F32, "f16": G.F16, "bf16": G.BF16}
TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
ODT = {"f32": O.F32, "f16": O.F16, "bf16": O.BF16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from activation_cnn_gb300 import build
    build.build()
    A.lib()
    yield
    torch.cuda.synchronize()
    assert A.acnn_last_device_status() == 0


def conv_case(name, n, h, w, cin, cout, k, s, p, dt, layout=G.NHWC, act=A.ACT_RELU,
              res_mode=A.RES_NONE, bias=True, integer=False, kw=None):
    kw = kw or k
    seed = 11
    xs = G.activation_shape(layout, n, cin, h, w)
    if integer:
        x = G.tensor(seed, name + ".x", xs, "int", -3, 3, dtype=DT[dt])
        wshape = (cout, k, kw, cin) if layout == G.NHWC else (cout, cin, k, kw)
        wt = G.tensor(seed, name + ".w", wshape, "int", -2, 2, dtype=DT[dt])
        b = G.tensor(seed, name + ".b", (cout,), "int", -4, 4) if bias else None
        al = torch.full((cout,), 0.25)
    else:
        x = G.tensor(seed, name + ".x", xs, "normal", dtype=DT[dt])
        wt = G.conv_weight(seed, name, cout, cin, k, kw, layout, DT[dt])
        b = G.conv_bias(seed, name, cout) if bias else None
        al = G.prelu_alpha(seed, name, cout)
    oh, ow = (h + 2 * p - k) // s + 1, (w + 2 * p - kw) // s + 1
    ys = G.activation_shape(layout, n, cout, oh, ow)
    r = G.tensor(seed, name + ".r", ys, "normal", dtype=DT[dt]) if res_mode else None
    dev = lambda t: None if t is None else t.cuda()
    # output and workspace inside canary guards (see tests.parity.Guarded)
    d = A.conv_desc(x, cout, k, kw, s, p, layout)
    gy = Guarded(A.conv_out_shape(d), TDT[dt])
    gws = guarded_bytes(A.acnn_conv2d_workspace_size(d))
    y = A.conv2d_fused(dev(x), dev(wt), dev(b), stride=s, pad=p, act=act, alpha=dev(al),
                       residual=dev(r), res_mode=res_mode, layout=layout, out=gy.t,
                       workspace=None if gws is None else gws.t)
    gy.check(name + " output")
    if gws is not None:
        gws.check(name + " workspace")
    ref = O.conv2d(to64(x), to64(wt), None if b is None else to64(b), stride=s, pad=p, act=act,
                   alpha=to64(al), residual=None if r is None else to64(r), res_mode=res_mode,
                   layout=layout)
    return y, ref


# ---------------------------------------------------------------- tensor-core path
TC_CASES = [
    # name, n, h, w, cin, cout, k, s, p
    ("1x1_tail", 2, 9, 11, 64, 64, 1, 1, 0),
    ("1x1_wide", 1, 16, 20, 256, 256, 1, 1, 0),
    ("1x1_cin128_cout512", 1, 12, 12, 128, 512, 1, 1, 0),
    ("1x1_cin32", 3, 7, 9, 32, 64, 1, 1, 0),
    ("1x1_cin8", 1, 10, 13, 8, 16, 1, 1, 0),
    ("3x3_s1", 2, 13, 17, 64, 64, 3, 1, 1),
    ("3x3_s2", 3, 15, 14, 64, 128, 3, 2, 1),
    ("3x3_s2_even", 2, 16, 16, 128, 128, 3, 2, 1),
    ("3x3_cout240", 1, 11, 19, 128, 240, 3, 1, 1),
    ("3x3_cin32", 2, 12, 12, 32, 32, 3, 1, 1),
    ("3x3_cin96", 1, 9, 9, 96, 48, 3, 1, 1),
    ("3x3_p0", 1, 10, 12, 64, 64, 3, 1, 0),
    ("5x5_s1", 1, 11, 10, 64, 64, 5, 1, 2),
    ("7x7_s2", 2, 19, 21, 16, 64, 7, 2, 3),
    ("1x1_s2", 2, 9, 10, 64, 64, 1, 2, 0),
    ("3x3_big_m", 2, 40, 41, 64, 64, 3, 1, 1),
    # C_in <= 32: 32-channel k-blocks (64-byte swizzle), BN = 32/64/128
    ("3x3_cin32_cout64_big", 2, 40, 37, 32, 64, 3, 1, 1),
    ("3x3_cin24_cout32", 1, 21, 23, 24, 32, 3, 1, 1),
    ("1x1_cin16_cout128", 1, 30, 30, 16, 128, 1, 1, 0),
    ("3x3_cin32_cout96", 1, 19, 22, 32, 96, 3, 1, 1),
    ("3x3_s2_cin8", 2, 33, 29, 8, 48, 3, 2, 1),
]


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("case", TC_CASES, ids=[c[0] for c in TC_CASES])
def test_conv_tensor_path(case, dt):
    name, n, h, w, cin, cout, k, s, p = case
    d = A.ConvDesc(n, h, w, cin, cout, k, k, s, p, G.NHWC, DT[dt])
    assert A.acnn_conv2d_path(d) in (1, 2)
    y, ref = conv_case(name, n, h, w, cin, cout, k, s, p, dt)
    assert_parity(y, ref, TDT[dt], name)


@pytest.mark.parametrize("act", [A.ACT_NONE, A.ACT_RELU, A.ACT_SILU, A.ACT_PRELU])
@pytest.mark.parametrize("res_mode", [A.RES_NONE, A.RES_ADD_THEN_ACT, A.RES_ACT_THEN_ADD])
def test_conv_tensor_epilogue_modes(act, res_mode):
    y, ref = conv_case(f"epi{act}{res_mode}", 2, 10, 14, 64, 128, 3, 1, 1, "bf16", act=act,
                       res_mode=res_mode)
    assert_parity(y, ref, torch.bfloat16, f"act{act} res{res_mode}")


# Several tiles per CTA (more tiles than SMs), so the epilogue's residual ring
# and its bias prefetch cross tile boundaries; a ragged second column tile
# (C_out = 96 with 64-wide tiles) in the second case.
@pytest.mark.parametrize("shape", [(4, 96, 96, 64, 256), (4, 64, 64, 64, 96), (2, 80, 80, 32, 64)])
@pytest.mark.parametrize("act,res_mode", [(A.ACT_RELU, A.RES_ADD_THEN_ACT),
                                          (A.ACT_PRELU, A.RES_ACT_THEN_ADD),
                                          (A.ACT_SILU, A.RES_NONE)])
def test_conv_tensor_multi_tile_epilogue(shape, act, res_mode):
    n, h, w, cin, cout = shape
    y, ref = conv_case(f"mt{shape}", n, h, w, cin, cout, 1, 1, 0, "bf16", act=act,
                       res_mode=res_mode)
    assert_parity(y, ref, torch.bfloat16, f"multi-tile {shape}")


@pytest.mark.parametrize("n,hw,cin,cout,k", [(80, 320, 256, 256, 1), (320, 320, 64, 64, 3)])
def test_conv_tensor_near_index_limit(n, hw, cin, cout, k):
    """Output maps of just under 2^31 elements (4.3 GB of bf16 each way): one
    seeded 320x320 image repeated n times, so every image's output equals the
    first's; sampled pixels across all images, the last pixel included, against
    the oracle on that one image (64-bit offsets in every load and store)."""
    name = f"big{k}"
    x1 = G.tensor(12, name + ".x", (1, hw, hw, cin), "normal", dtype=G.BF16)
    wt = G.conv_weight(12, name, cout, cin, k, k, G.NHWC, G.BF16)
    b = G.conv_bias(12, name, cout)
    assert n * hw * hw * cout < 2**31 and n * hw * hw * cout > 2**31 - 2**28
    x = x1.cuda().expand(n, hw, hw, cin).contiguous()
    y = A.conv2d_fused(x, wt.cuda(), b.cuda(), stride=1, pad=k // 2, act=A.ACT_RELU)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    pts = [(n - 1, hw - 1, hw - 1), (0, 0, 0), (n // 2, 0, hw - 1), (n - 1, 0, 0)]
    pts += [(int(rng.integers(n)), int(rng.integers(hw)), int(rng.integers(hw))) for _ in range(60)]
    got = torch.stack([y[i, oy, ox] for i, oy, ox in pts]).cpu()
    ref = O.conv2d_points(to64(x1), to64(wt), to64(b), [(0, oy, ox) for _, oy, ox in pts],
                          stride=1, pad=k // 2, act=A.ACT_RELU)
    del x, y
    torch.cuda.empty_cache()
    assert_parity(got, ref, torch.bfloat16, name)


PREPACK_CASES = [
    # name, layout, dtype, n, h, w, cin, cout, k, s, p, act
    ("nchw_3x3", G.NCHW, "f16", 1, 17, 30, 120, 240, 3, 1, 1, A.ACT_PRELU),
    ("nchw_packed_7", G.NCHW, "f16", 1, 36, 52, 7, 120, 3, 2, 1, A.ACT_PRELU),
    ("nhwc_packed_rgb", G.NHWC, "bf16", 2, 40, 48, 3, 32, 3, 2, 1, A.ACT_RELU),
    ("nhwc_3x3", G.NHWC, "bf16", 2, 13, 17, 64, 64, 3, 1, 1, A.ACT_SILU),
    ("nchw_1x1", G.NCHW, "f16", 1, 9, 15, 240, 64, 1, 1, 0, A.ACT_RELU),
    ("f32_direct", G.NHWC, "f32", 1, 12, 12, 16, 32, 3, 1, 1, A.ACT_RELU),
]


@pytest.mark.parametrize("case", PREPACK_CASES, ids=[c[0] for c in PREPACK_CASES])
def test_conv_prepacked_equals_plain(case):
    """Prepacked weights give the same bits as the per-call staging, on every
    path (direct, tiled, im2col, packed; NHWC and NCHW), and match the oracle."""
    name, layout, dt, n, h, w, cin, cout, k, s, p, act = case
    seed = 13
    x = G.tensor(seed, name + ".x", G.activation_shape(layout, n, cin, h, w), "normal",
                 dtype=DT[dt]).cuda()
    wt = G.conv_weight(seed, name, cout, cin, k, k, layout, DT[dt]).cuda()
    b = G.conv_bias(seed, name, cout).cuda()
    al = G.prelu_alpha(seed, name, cout).cuda()
    y = A.conv2d_fused(x, wt, b, stride=s, pad=p, act=act, alpha=al, layout=layout)
    d = A.conv_desc(x, cout, k, k, s, p, layout)
    wp = A.conv2d_prepack(d, wt)
    wsb = A.acnn_conv2d_prepacked_workspace_size(d)
    assert wsb <= A.acnn_conv2d_workspace_size(d)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    y2 = torch.empty_like(y)
    A.check(A.acnn_conv2d_fused_prepacked(d, x, wp, b, al, None, A.RES_NONE, act, y2, ws, wsb,
                                          None), name)
    torch.cuda.synchronize()
    assert torch.equal(y, y2), name
    ref = O.conv2d(to64(x), to64(wt), to64(b), stride=s, pad=p, act=act, alpha=to64(al),
                   layout=layout)
    assert_parity(y2, ref, TDT[dt], name)


@pytest.mark.parametrize("layout", [G.NHWC, G.NCHW])
def test_conv_tiny_prepacked_equals_plain(layout, tiny_path):
    """On the direct tiny-C_in kernel the prepacked weights are an unchanged copy."""
    dt = "f16"
    x = G.tensor(14, "tpp.x", G.activation_shape(layout, 1, 7, 30, 44), "normal",
                 dtype=DT[dt]).cuda()
    wt = G.conv_weight(14, "tpp", 48, 7, 3, 3, layout, DT[dt]).cuda()
    b = G.conv_bias(14, "tpp", 48).cuda()
    y = A.conv2d_fused(x, wt, b, stride=2, pad=1, act=A.ACT_RELU, layout=layout)
    d = A.conv_desc(x, 48, 3, 3, 2, 1, layout)
    assert A.acnn_conv2d_path(d) == 4
    wp = A.conv2d_prepack(d, wt)
    y2 = torch.empty_like(y)
    A.check(A.acnn_conv2d_fused_prepacked(d, x, wp, b, None, None, A.RES_NONE, A.ACT_RELU, y2,
                                          None, 0, None), "tiny prepacked")
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


@pytest.mark.parametrize("case", [(1, 17, 30, 120, 240, 2, A.RES_NONE, 3),
                                  (1, 9, 15, 240, 240, 1, A.RES_ACT_THEN_ADD, 3),
                                  (2, 8, 8, 64, 32, 1, A.RES_NONE, 3),
                                  (1, 34, 60, 7, 120, 2, A.RES_NONE, 3),      # packed path
                                  (1, 13, 21, 96, 64, 1, A.RES_ADD_THEN_ACT, 1)])
def test_conv_nchw_staged_copies(case):
    """NCHW conv with an NHWC copy of its input supplied and/or of its output
    written (acnn_conv2d_fused_prepacked_staged): y bit-identical to the plain
    prepacked call, the output copy equal to y in NHWC, nothing written outside
    either; the input copy spares the staging (a workspace without it works)."""
    n, h, w, cin, cout, s_, res_mode, k = case
    dt = "f16"
    seed = 17
    x = G.tensor(seed, "stc.x", (n, cin, h, w), "normal", dtype=DT[dt]).cuda()
    wt = G.conv_weight(seed, "stc", cout, cin, k, k, G.NCHW, DT[dt]).cuda()
    b = G.conv_bias(seed, "stc", cout).cuda()
    al = G.prelu_alpha(seed, "stc", cout).cuda()
    p_ = k // 2
    d = A.conv_desc(x, cout, k, k, s_, p_, G.NCHW)
    oh, ow = (h + 2 * p_ - k) // s_ + 1, (w + 2 * p_ - k) // s_ + 1
    r = G.tensor(seed, "stc.r", (n, cout, oh, ow), "normal", dtype=DT[dt]).cuda() if res_mode else None
    wp = A.conv2d_prepack(d, wt)
    wsb = A.acnn_conv2d_prepacked_workspace_size(d)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    y_ref = torch.empty((n, cout, oh, ow), dtype=torch.float16, device="cuda")
    A.check(A.acnn_conv2d_fused_prepacked(d, x, wp, b, al, r, res_mode, A.ACT_PRELU, y_ref, ws,
                                          wsb, None), "plain")
    path = A.acnn_conv2d_path(d)
    x_copy = x.permute(0, 2, 3, 1).contiguous() if path in (1, 2) else None
    gy = Guarded((n, cout, oh, ow), torch.float16)
    gc = Guarded((n, oh, ow, cout), torch.float16)
    # with the input copy the staging part of the workspace is not needed
    st = A.acnn_conv2d_fused_prepacked_staged(d, x, x_copy, wp, b, al, r, res_mode, A.ACT_PRELU,
                                              gy.t, gc.t, ws if x_copy is None else None,
                                              wsb if x_copy is None else 0)
    assert st == 0, A.status_string(st)
    gy.check("staged y")
    gc.check("staged y copy")
    torch.cuda.synchronize()
    assert_bitexact(gy.t, y_ref, f"staged y {case}")
    assert_bitexact(gc.t, y_ref.permute(0, 2, 3, 1).contiguous(), f"staged copy {case}")


def test_conv_staged_copies_rejected():
    """Copies only for NCHW convs on the tensor-core paths (input copy: paths 1-2)."""
    X, W, Y, C = (torch.empty(1 << 20, dtype=torch.uint8, device="cuda") for _ in range(4))
    nhwc = A.ConvDesc(1, 8, 8, 64, 64, 3, 3, 1, 1, G.NHWC, G.F16)
    assert A.acnn_conv2d_fused_prepacked_staged(nhwc, X, C, W, None, None, None, 0, 0, Y, None,
                                                None, 0) == 3
    f32 = A.ConvDesc(1, 8, 8, 16, 32, 3, 3, 1, 1, G.NCHW, G.F32)
    assert A.acnn_conv2d_fused_prepacked_staged(f32, X, None, W, None, None, None, 0, 0, Y, C,
                                                None, 0) == 3
    packed = A.ConvDesc(1, 8, 8, 7, 64, 3, 3, 1, 1, G.NCHW, G.F16)
    assert A.acnn_conv2d_fused_prepacked_staged(packed, X, C, W, None, None, None, 0, 0, Y, None,
                                                None, 0) == 3


def test_conv_tensor_no_bias():
    y, ref = conv_case("nobias", 1, 9, 9, 64, 64, 1, 1, 0, "f16", bias=False)
    assert_parity(y, ref, torch.float16)


@pytest.mark.parametrize("k,s,p", [(1, 1, 0), (3, 1, 1), (3, 2, 1)])
def test_conv_tensor_integer_bitexact(k, s, p):
    """Integer data: fp32 sums are exact, so the bf16 store equals RNE of the oracle."""
    y, ref = conv_case(f"int{k}{s}", 2, 11, 13, 64, 64, k, s, p, "bf16", act=A.ACT_PRELU,
                       integer=True)
    assert_bitexact(y, O.round_storage(ref, O.BF16), f"int k{k} s{s}")


@pytest.mark.parametrize("act,res_mode", [(A.ACT_PRELU, A.RES_ACT_THEN_ADD),
                                          (A.ACT_RELU, A.RES_ADD_THEN_ACT),
                                          (A.ACT_NONE, A.RES_NONE)])
@pytest.mark.parametrize("shape", [(1, 17, 30, 120, 240, 2), (1, 9, 15, 240, 240, 1),
                                   (2, 8, 8, 64, 32, 1),
                                   # output planes of 8k pixels: the vectorised
                                   # stores, with chunks inside one image (384)
                                   # and straddling two (40), ragged C_out (72)
                                   (1, 16, 24, 120, 240, 1), (3, 5, 8, 64, 72, 1),
                                   (1, 68, 120, 240, 240, 1)])
def test_conv_tensor_nchw(shape, act, res_mode):
    """NCHW fp16 on the tensor path (workspace transpose + NCHW-writing epilogue)."""
    n, h, w, cin, cout, s = shape
    d = A.ConvDesc(n, h, w, cin, cout, 3, 3, s, 1, G.NCHW, G.F16)
    assert A.acnn_conv2d_path(d) == 2 and A.acnn_conv2d_workspace_size(d) > 0
    y, ref = conv_case(f"nchw{shape}", n, h, w, cin, cout, 3, s, 1, "f16", layout=G.NCHW,
                       act=act, res_mode=res_mode)
    assert_parity(y, ref, torch.float16, f"nchw {shape}")


def test_conv_tensor_repeat_is_deterministic():
    name = "repeat"
    x = G.tensor(1, name + ".x", (2, 20, 20, 64), "normal", dtype=G.BF16).cuda()
    wt = G.conv_weight(1, name, 128, 64, 3, 3, G.NHWC, G.BF16).cuda()
    a = A.conv2d_fused(x, wt, None, pad=1)
    b = A.conv2d_fused(x, wt, None, pad=1)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# ---------------------------------------------------------------- direct path
DIRECT_CASES = [
    # name, n, h, w, cin, cout, k, s, p, dt, layout
    ("cfg1_like", 1, 32, 32, 16, 32, 3, 1, 1, "f32", G.NHWC),
    ("stem_s2_f32", 1, 37, 45, 3, 32, 3, 2, 1, "f32", G.NHWC),
    ("f32_32to64", 1, 21, 19, 32, 64, 3, 1, 1, "f32", G.NHWC),
    ("f32_nchw", 2, 15, 17, 5, 20, 3, 1, 1, "f32", G.NCHW),
    ("f32_7x7", 1, 23, 18, 3, 40, 7, 2, 3, "f32", G.NHWC),
    ("f32_1x1", 1, 10, 10, 12, 36, 1, 1, 0, "f32", G.NHWC),
    ("f16_cout_odd", 1, 12, 12, 24, 30, 3, 1, 1, "f16", G.NHWC),
    ("f32_5x5_s3", 1, 20, 26, 6, 33, 5, 3, 2, "f32", G.NHWC),
]


@pytest.mark.parametrize("case", DIRECT_CASES, ids=[c[0] for c in DIRECT_CASES])
def test_conv_direct_path(case):
    name, n, h, w, cin, cout, k, s, p, dt, layout = case
    d = A.ConvDesc(n, h, w, cin, cout, k, k, s, p, layout, DT[dt])
    assert A.acnn_conv2d_path(d) == 0
    y, ref = conv_case(name, n, h, w, cin, cout, k, s, p, dt, layout=layout)
    assert_parity(y, ref, TDT[dt], name)


PACKED_CASES = [
    # name, n, h, w, cin, cout, k, kw, s, p, dt, layout
    ("stem_s2_bf16", 2, 33, 30, 3, 32, 3, 3, 2, 1, "bf16", G.NHWC),
    ("stem_s2_big", 2, 160, 150, 3, 32, 3, 3, 2, 1, "bf16", G.NHWC),
    ("prep7_nchw_f16", 1, 34, 60, 7, 120, 3, 3, 2, 1, "f16", G.NCHW),
    ("cin5_7x7_s2", 1, 41, 37, 5, 64, 7, 7, 2, 3, "bf16", G.NHWC),
    ("cin5_3x3_s2", 2, 33, 30, 5, 32, 3, 3, 2, 1, "bf16", G.NHWC),
    ("nonsq_1x3", 2, 12, 17, 16, 48, 1, 3, 1, 0, "f16", G.NHWC),
    ("cin12_3x3", 1, 23, 29, 12, 40, 3, 3, 1, 1, "bf16", G.NCHW),
]


@pytest.mark.parametrize("case", PACKED_CASES, ids=[c[0] for c in PACKED_CASES])
def test_conv_packed_path(case):
    """Few/odd input channels or non-square kernels: explicit im2col pack + tcgen05 GEMM."""
    name, n, h, w, cin, cout, k, kw, s, p, dt, layout = case
    d = A.ConvDesc(n, h, w, cin, cout, k, kw, s, p, layout, DT[dt])
    assert A.acnn_conv2d_path(d) == 3
    y, ref = conv_case(name, n, h, w, cin, cout, k, s, p, dt, layout=layout, kw=kw)
    assert_parity(y, ref, TDT[dt], name)


# ---------------------------------------------------------------- halo rows
# 3x3 stride-1 pad-1 convs run on a virtual output grid two columns wider than
# the map (one box of 128 + 2 pixels per kernel row serves its three horizontal
# taps; the two extra columns of each row are computed and discarded): widths
# where those columns are most of a row, tiles straddling rows and images,
# 32- and 64-channel k-blocks, both layouts, residual modes.
HALO_CASES = [
    # name, n, h, w, cin, cout, layout, res_mode
    ("w1", 3, 7, 1, 64, 64, G.NHWC, A.RES_NONE),
    ("w2", 2, 9, 2, 64, 128, G.NHWC, A.RES_ADD_THEN_ACT),
    ("w3_cin32", 4, 5, 3, 32, 64, G.NHWC, A.RES_NONE),
    ("w126", 1, 3, 126, 64, 64, G.NHWC, A.RES_ACT_THEN_ADD),  # vw = 128: rows on tile edges
    ("w127_cin32", 2, 4, 127, 32, 32, G.NHWC, A.RES_NONE),
    ("h1", 5, 1, 37, 128, 64, G.NHWC, A.RES_NONE),
    ("nchw_w5", 2, 11, 5, 64, 48, G.NCHW, A.RES_ACT_THEN_ADD),
    ("nchw_w120", 1, 9, 120, 240, 240, G.NCHW, A.RES_NONE),
    ("cin96", 3, 13, 29, 96, 64, G.NHWC, A.RES_ADD_THEN_ACT),
]


@pytest.mark.parametrize("case", HALO_CASES, ids=[c[0] for c in HALO_CASES])
def test_conv_halo_rows(case):
    name, n, h, w, cin, cout, layout, res_mode = case
    dt = "bf16" if layout == G.NHWC else "f16"
    d = A.ConvDesc(n, h, w, cin, cout, 3, 3, 1, 1, layout, DT[dt])
    assert A.acnn_conv2d_path(d) == 2
    y, ref = conv_case("halo" + name, n, h, w, cin, cout, 3, 1, 1, dt, layout=layout,
                       act=A.ACT_PRELU, res_mode=res_mode)
    assert_parity(y, ref, TDT[dt], name)


@pytest.mark.parametrize("cin", [32, 64])
def test_conv_halo_rows_integer_bitexact(cin):
    """Integer data on the halo-row path: every product and partial sum exact, so
    each stored value is the oracle's rounded once (a tap read from the wrong
    row or column of the box would change it)."""
    y, ref = conv_case(f"hint{cin}", 2, 15, 23, cin, 64, 3, 1, 1, "bf16", act=A.ACT_PRELU,
                       integer=True)
    assert_bitexact(y, O.round_storage(ref, O.BF16), f"halo int cin{cin}")


# ---------------------------------------------------------------- conv + pooled output
POOL2_CASES = [
    # name, n, h, w, cin, cout, act, res_mode
    ("s1_like", 2, 16, 32, 64, 256, A.ACT_RELU, A.RES_ADD_THEN_ACT),      # 16 x 8 tiles
    ("s3_like", 2, 40, 40, 256, 512, A.ACT_RELU, A.RES_ADD_THEN_ACT),     # 8 x 16, rows ragged
    ("ragged_both", 1, 6, 10, 128, 64, A.ACT_SILU, A.RES_NONE),          # neither divides
    ("w24", 3, 20, 24, 64, 128, A.ACT_PRELU, A.RES_ACT_THEN_ADD),
    ("one_window", 1, 2, 2, 64, 64, A.ACT_NONE, A.RES_NONE),
    ("cout72", 2, 8, 16, 96, 72, A.ACT_RELU, A.RES_NONE),                # ragged column tile
]


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("case", POOL2_CASES, ids=[c[0] for c in POOL2_CASES])
def test_conv_fused_pool2(case, dt):
    """The 1x1 conv with a pooled second output: y bit-identical to acnn_conv2d_fused,
    y_pool bit-identical to acnn_pool2d (average 2x2/s2) of y, both within
    tolerance of the oracle, nothing written outside either buffer."""
    name, n, h, w, cin, cout, act, res_mode = case
    seed = 15
    x = G.tensor(seed, name + ".x", (n, h, w, cin), "normal", dtype=DT[dt]).cuda()
    wt = G.conv_weight(seed, name, cout, cin, 1, 1, G.NHWC, DT[dt]).cuda()
    b = G.conv_bias(seed, name, cout).cuda()
    al = G.prelu_alpha(seed, name, cout).cuda()
    r = G.tensor(seed, name + ".r", (n, h, w, cout), "normal", dtype=DT[dt]).cuda() \
        if res_mode else None
    gy = Guarded((n, h, w, cout), TDT[dt])
    gp = Guarded((n, h // 2, w // 2, cout), TDT[dt])
    d = A.conv_desc(x, cout, 1, 1, 1, 0, G.NHWC)
    st = A.acnn_conv2d_fused_pool2(d, x, wt, b, al, r, res_mode, act, gy.t, gp.t)
    assert st == 0, A.status_string(st)
    gy.check(name + " y")
    gp.check(name + " y_pool")
    y_ref = A.conv2d_fused(x, wt, b, act=act, alpha=al, residual=r, res_mode=res_mode)
    p_ref = A.pool2d(y_ref, A.POOL_AVG, 2, 2, 0)
    torch.cuda.synchronize()
    assert_bitexact(gy.t, y_ref, name + " y vs conv2d_fused")
    assert_bitexact(gp.t, p_ref, name + " y_pool vs pool2d")
    ref = O.conv2d(to64(x), to64(wt), to64(b), act=act, alpha=to64(al),
                   residual=None if r is None else to64(r), res_mode=res_mode)
    assert_parity(gy.t, ref, TDT[dt], name)
    # the oracle pools the stored (rounded) conv output, as the workloads do
    ref_p = O.pool2d(O.round_storage(ref, ODT[dt]), O.AVG, 2, 2, 0)
    assert_parity(gp.t, ref_p, TDT[dt], name + " pooled")


UP2_CASES = [
    # name, n, h, w, c_a, c_b, cout, k, act, res_mode
    ("lat5_like", 8, 20, 20, 2048, 0, 256, 1, A.ACT_SILU, A.RES_NONE),      # split K
    ("fpn4_like", 2, 40, 40, 256, 256, 256, 3, A.ACT_SILU, A.RES_NONE),     # folded concat
    ("odd", 1, 5, 7, 64, 0, 64, 3, A.ACT_RELU, A.RES_ADD_THEN_ACT),
    ("csp_out", 2, 10, 12, 256, 256, 256, 1, A.ACT_SILU, A.RES_ACT_THEN_ADD),
]


@pytest.mark.parametrize("case", UP2_CASES, ids=[c[0] for c in UP2_CASES])
def test_conv_fused_up2(case):
    """A conv that also writes the nearest 2x upsample of its output: y bit-identical
    to the plain (or concat-folded) conv, y_up bit-identical to resize2d nearest of y,
    nothing written outside either buffer."""
    name, n, h, w, ca, cb, cout, k, act, res_mode = case
    seed, dt = 16, "bf16"
    cin = ca + cb
    xa = G.tensor(seed, name + ".xa", (n, h, w, ca), "normal", dtype=DT[dt]).cuda()
    xb = G.tensor(seed, name + ".xb", (n, h, w, cb), "normal", dtype=DT[dt]).cuda() if cb else None
    wt = G.conv_weight(seed, name, cout, cin, k, k, G.NHWC, DT[dt]).cuda()
    b = G.conv_bias(seed, name, cout).cuda()
    r = G.tensor(seed, name + ".r", (n, h, w, cout), "normal", dtype=DT[dt]).cuda() \
        if res_mode else None
    d = A.ConvDesc(n, h, w, cin, cout, k, k, 1, k // 2, G.NHWC, DT[dt])
    ws_bytes = A.acnn_conv2d_workspace_size(d)
    gws = guarded_bytes(ws_bytes)
    gy = Guarded((n, h, w, cout), TDT[dt])
    gu = Guarded((n, 2 * h, 2 * w, cout), TDT[dt])
    st = A.acnn_conv2d_fused_up2(d, xa, ca, xb, wt, b, None, r, res_mode, act, gy.t, gu.t,
                                 None if gws is None else gws.t, ws_bytes)
    assert st == 0, A.status_string(st)
    gy.check(name + " y")
    gu.check(name + " y_up")
    if gws is not None:
        gws.check(name + " workspace")
    if xb is None:
        y_ref = A.conv2d_fused(xa, wt, b, pad=k // 2, act=act, residual=r, res_mode=res_mode)
    else:
        y_ref = A.conv2d_fused_cat2(xa, xb, wt, b, pad=k // 2, act=act, residual=r,
                                    res_mode=res_mode)
    u_ref = A.resize2d(y_ref, A.RESIZE_NEAREST, 2 * h, 2 * w)
    torch.cuda.synchronize()
    assert_bitexact(gy.t, y_ref, name + " y")
    assert_bitexact(gu.t, u_ref, name + " y_up")
    x64 = to64(xa) if xb is None else O.concat(to64(xa), to64(xb))
    ref = O.conv2d(x64, to64(wt), to64(b), pad=k // 2, act=act,
                   residual=None if r is None else to64(r), res_mode=res_mode)
    assert_parity(gy.t, ref, TDT[dt], name)


def test_conv_fused_pool2_rejects():
    """Only 1x1/s1/p0 NHWC 16-bit convs with C_in >= 64 and an even output map."""
    X, W, Y, P = (torch.empty(4 << 20, dtype=torch.uint8, device="cuda") for _ in range(4))
    for desc in (A.ConvDesc(1, 8, 8, 64, 64, 3, 3, 1, 1, G.NHWC, G.BF16),   # 3x3
                 A.ConvDesc(1, 7, 8, 64, 64, 1, 1, 1, 0, G.NHWC, G.BF16),   # odd height
                 A.ConvDesc(1, 8, 8, 32, 64, 1, 1, 1, 0, G.NHWC, G.BF16),   # 32-channel blocks
                 A.ConvDesc(1, 8, 8, 64, 64, 1, 1, 1, 0, G.NCHW, G.F16),    # NCHW
                 A.ConvDesc(1, 8, 8, 64, 64, 1, 1, 1, 0, G.NHWC, G.F32)):   # fp32
        st = A.acnn_conv2d_fused_pool2(desc, X, W, None, None, None, 0, 0, Y, P)
        assert st == 3, A.status_string(st)  # ACNN_ERR_UNSUPPORTED
    d = A.ConvDesc(1, 8, 8, 64, 64, 1, 1, 1, 0, G.NHWC, G.BF16)
    assert A.acnn_conv2d_fused_pool2(d, X, W, None, None, None, 0, 0, Y, None) == 1
    assert A.acnn_conv2d_fused_pool2(d, X, W, None, None, None, 0, 0, Y, Y) == 6  # alias


# ---------------------------------------------------------------- tiny C_in (path 4)
TINY_CASES = [
    # name, n, h, w, cin, cout, s, p, dt, layout
    ("stem_rgb", 2, 33, 30, 3, 32, 2, 1, "bf16", G.NHWC),
    ("stem_rgb_big", 2, 160, 150, 3, 32, 2, 1, "bf16", G.NHWC),
    ("stem_rgb_f16", 1, 64, 66, 3, 32, 2, 1, "f16", G.NHWC),
    ("frame7", 1, 34, 60, 7, 120, 2, 1, "f16", G.NCHW),
    ("frame7_bf16", 1, 36, 44, 7, 120, 2, 1, "bf16", G.NCHW),
    ("frame6", 1, 68, 120, 6, 120, 2, 1, "f16", G.NCHW),
    ("s1_nhwc", 2, 21, 37, 3, 40, 1, 1, "bf16", G.NHWC),   # ragged channel chunk
    ("s1_nchw", 1, 19, 45, 7, 24, 1, 1, "f16", G.NCHW),    # OW % 4 != 0: scalar stores
    ("nhwc_cout12", 1, 17, 29, 3, 12, 2, 1, "bf16", G.NHWC),  # C_out % 8 != 0
    ("p0_s2", 2, 23, 41, 6, 64, 2, 0, "f16", G.NCHW),
    ("p2_s1", 1, 9, 12, 7, 16, 1, 2, "bf16", G.NHWC),
    ("one_px", 3, 1, 1, 3, 8, 1, 1, "bf16", G.NHWC),
]


@pytest.fixture(params=[0, 1], ids=["smem_weights", "shfl_weights"])
def tiny_path(request):
    """Route the tiny-C_in geometries to the direct kernel (the router prefers the
    packed path for them), with weights broadcast from shared memory or by warp
    shuffles."""
    assert A.acnn_conv2d_force_path(4, request.param) == 0
    yield request.param
    assert A.acnn_conv2d_force_path(0, 0) == 0


@pytest.mark.parametrize("case", TINY_CASES, ids=[c[0] for c in TINY_CASES])
def test_conv_tiny_path(case, tiny_path):
    """3, 6 or 7 input channels, fp16/bf16, 3x3: the direct kernel with the input
    patch in shared memory."""
    name, n, h, w, cin, cout, s, p, dt, layout = case
    d = A.ConvDesc(n, h, w, cin, cout, 3, 3, s, p, layout, DT[dt])
    assert A.acnn_conv2d_path(d) == 4 and A.acnn_conv2d_workspace_size(d) == 0
    y, ref = conv_case("tiny" + name, n, h, w, cin, cout, 3, s, p, dt, layout=layout,
                       act=A.ACT_PRELU if layout == G.NCHW else A.ACT_RELU)
    assert_parity(y, ref, TDT[dt], name)


@pytest.mark.parametrize("act", [A.ACT_NONE, A.ACT_RELU, A.ACT_SILU, A.ACT_PRELU])
@pytest.mark.parametrize("res_mode", [A.RES_NONE, A.RES_ADD_THEN_ACT, A.RES_ACT_THEN_ADD])
@pytest.mark.parametrize("layout", [G.NHWC, G.NCHW])
def test_conv_tiny_epilogue_modes(act, res_mode, layout, tiny_path):
    y, ref = conv_case(f"tepi{act}{res_mode}{layout}", 2, 18, 36, 7, 40, 3, 2, 1, "f16",
                       layout=layout, act=act, res_mode=res_mode)
    assert_parity(y, ref, torch.float16, f"tiny act{act} res{res_mode} layout{layout}")


@pytest.mark.parametrize("layout", [G.NHWC, G.NCHW])
@pytest.mark.parametrize("s", [1, 2])
def test_conv_tiny_integer_bitexact(layout, s, tiny_path):
    """Integer data: every fp32 partial sum is exact, so the stored value is the
    oracle's rounded once."""
    y, ref = conv_case(f"tint{layout}{s}", 2, 19, 26, 7, 48, 3, s, 1, "bf16", layout=layout,
                       act=A.ACT_PRELU, integer=True)
    assert_bitexact(y, O.round_storage(ref, O.BF16), f"tiny int layout{layout} s{s}")


def test_conv_direct_nonsquare():
    y, ref = conv_case("nonsq", 1, 12, 14, 4, 8, 1, 1, 0, "f32", kw=3)
    assert_parity(y, ref, torch.float32)


@pytest.mark.parametrize("act", [A.ACT_SILU, A.ACT_PRELU])
@pytest.mark.parametrize("res_mode", [A.RES_ADD_THEN_ACT, A.RES_ACT_THEN_ADD])
def test_conv_direct_epilogue_modes(act, res_mode):
    y, ref = conv_case(f"depi{act}{res_mode}", 1, 20, 21, 8, 16, 3, 1, 1, "f32", act=act,
                       res_mode=res_mode)
    assert_parity(y, ref, torch.float32)


def test_conv_direct_integer_bitexact_f32():
    y, ref = conv_case("dint", 2, 19, 23, 16, 32, 3, 1, 1, "f32", act=A.ACT_PRELU, integer=True)
    assert_bitexact(y, ref)


# ---------------------------------------------------------------- pools
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("layout", [G.NHWC, G.NCHW])
@pytest.mark.parametrize("shape", [(2, 17, 23, 64), (1, 8, 8, 3), (3, 1, 1, 16), (1, 2, 5, 24),
                                   (1, 65, 129, 64)])
def test_maxpool_bitexact(dt, layout, shape):
    n, h, w, c = shape
    x = G.tensor(3, f"mp{shape}", G.activation_shape(layout, n, c, h, w), "normal", dtype=DT[dt])
    ref = O.pool2d(to64(x), O.MAX, 3, 2, 1, layout=layout)
    g = Guarded(ref.shape, TDT[dt])
    y = A.pool2d(x.cuda(), A.POOL_MAX, 3, 2, 1, layout=layout, out=g.t)
    g.check(f"maxpool {dt} {shape}")
    assert_bitexact(y, ref, f"{dt} {shape}")


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("layout", [G.NHWC, G.NCHW])
@pytest.mark.parametrize("shape", [(2, 16, 22, 64), (1, 8, 6, 5), (2, 33, 47, 256)])
def test_avgpool(dt, layout, shape):
    n, h, w, c = shape
    x = G.tensor(4, f"ap{shape}", G.activation_shape(layout, n, c, h, w), "normal", dtype=DT[dt])
    ref = O.pool2d(to64(x), O.AVG, 2, 2, 0, layout=layout)
    g = Guarded(ref.shape, TDT[dt])
    y = A.pool2d(x.cuda(), A.POOL_AVG, 2, 2, 0, layout=layout, out=g.t)
    g.check(f"avgpool {dt} {shape}")
    assert_parity(y, ref, TDT[dt])


def test_avgpool_integer_bitexact():
    x = G.tensor(4, "api", (2, 10, 12, 16), "int", -8, 8, dtype=G.BF16)
    y = A.pool2d(x.cuda(), A.POOL_AVG, 2, 2, 0)
    torch.cuda.synchronize()
    assert_bitexact(y, O.round_storage(O.pool2d(to64(x), O.AVG, 2, 2, 0), O.BF16))


# ---------------------------------------------------------------- resize
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("layout", [G.NHWC, G.NCHW])
@pytest.mark.parametrize("io", [((5, 7), (10, 14)), ((20, 20), (40, 40)), ((3, 5), (7, 11))])
def test_nearest_bitexact(dt, layout, io):
    (h, w), (oh, ow) = io
    x = G.tensor(5, f"nn{io}", G.activation_shape(layout, 2, 24, h, w), "normal", dtype=DT[dt])
    ref = O.resize2d(to64(x), O.NEAREST, oh, ow, layout=layout)
    g = Guarded(ref.shape, TDT[dt])
    y = A.resize2d(x.cuda(), A.RESIZE_NEAREST, oh, ow, layout=layout, out=g.t)
    g.check(f"nearest {dt} {io}")
    assert_bitexact(y, ref)


@pytest.mark.parametrize("dt_in,dt_out", [("f32", "f32"), ("f16", "f16"), ("bf16", "bf16"),
                                          ("f16", "f32")])
@pytest.mark.parametrize("layout", [G.NHWC, G.NCHW])
@pytest.mark.parametrize("io", [((16, 24), (4, 6)), ((9, 15), (72, 120)), ((7, 9), (5, 13))])
def test_bilinear(dt_in, dt_out, layout, io):
    (h, w), (oh, ow) = io
    x = G.tensor(6, f"bl{io}", G.activation_shape(layout, 2, 8, h, w), "normal", dtype=DT[dt_in])
    ref = O.resize2d(to64(x), O.BILINEAR, oh, ow, layout=layout)
    g = Guarded(ref.shape, TDT[dt_out])
    y = A.resize2d(x.cuda(), A.RESIZE_BILINEAR, oh, ow, layout=layout, out_dtype=TDT[dt_out],
                   out=g.t)
    g.check(f"bilinear {dt_in}->{dt_out} {io}")
    assert_parity(y, ref, TDT[dt_out])


# ---------------------------------------------------------------- concat
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [G.NHWC, G.NCHW])
@pytest.mark.parametrize("cc", [(256, 256), (3, 5), (64, 8)])
def test_concat_bitexact(dt, layout, cc):
    ca, cb = cc
    a = G.tensor(7, f"ca{cc}", G.activation_shape(layout, 2, ca, 9, 11), "normal", dtype=DT[dt])
    b = G.tensor(7, f"cb{cc}", G.activation_shape(layout, 2, cb, 9, 11), "normal", dtype=DT[dt])
    ref = O.concat(to64(a), to64(b), layout=layout)
    g = Guarded(ref.shape, TDT[dt])
    y = A.concat(a.cuda(), b.cuda(), layout=layout, out=g.t)
    g.check(f"concat {dt} {cc}")
    assert_bitexact(y, ref)


# ---------------------------------------------------------------- deconv
@pytest.mark.parametrize("dt_in,dt_out", [("f16", "f16"), ("f32", "f32"), ("bf16", "f32")])
@pytest.mark.parametrize("layout", [G.NCHW, G.NHWC])
@pytest.mark.parametrize("shape", [(2, 24, 5, 7, 9), (1, 240, 5, 68, 120), (1, 40, 20, 11, 70)])
def test_deconv(dt_in, dt_out, layout, shape):
    n, ci, co, h, w = shape
    x = G.tensor(8, "dcx", G.activation_shape(layout, n, ci, h, w), "normal", dtype=DT[dt_in])
    wt = G.deconv_weight(8, "dc", ci, co, 4)
    b = G.conv_bias(8, "dc", co)
    ref = O.deconv2d(to64(x), to64(wt), to64(b), layout=layout)
    g = Guarded(ref.shape, TDT[dt_out])
    y = A.deconv2d(x.cuda(), wt.cuda(), b.cuda(), layout=layout, out_dtype=TDT[dt_out], out=g.t)
    g.check(f"deconv {shape}")
    assert_parity(y, ref, TDT[dt_out])


@pytest.mark.parametrize("dt", ["f16"])
@pytest.mark.parametrize("layout", [G.NCHW, G.NHWC])
@pytest.mark.parametrize("shape", [(2, 24, 5, 7, 9), (1, 240, 5, 68, 120), (1, 40, 20, 11, 70),
                                   (3, 64, 3, 1, 1)])
def test_deconv_tensor_core(dt, layout, shape):
    """The 4x4/s2/p1 deconv regrouped as a 3x3 conv to 4 c_out channels on the
    tensor cores, then a pixel shuffle (acnn_deconv2d_ws): within tolerance of the
    oracle (whose weights stay fp32; here they are rounded to the storage type),
    nothing written outside the output or the workspace; the PReLU path too."""
    n, ci, co, h, w = shape
    x = G.tensor(8, "dcx", G.activation_shape(layout, n, ci, h, w), "normal", dtype=DT[dt])
    wt = G.deconv_weight(8, "dc", ci, co, 4)
    b = G.conv_bias(8, "dc", co)
    al = G.prelu_alpha(8, "dc", co)
    d = A.ConvDesc(n, h, w, ci, co, 4, 4, 2, 1, layout, DT[dt])
    ws_bytes = A.acnn_deconv2d_workspace_size(d, DT[dt])
    assert ws_bytes > 0
    gws = guarded_bytes(ws_bytes)
    for act in (A.ACT_NONE, A.ACT_PRELU):
        ref = O.deconv2d(to64(x), to64(wt), to64(b), layout=layout, act=act, alpha=to64(al))
        g = Guarded(ref.shape, TDT[dt])
        st = A.acnn_deconv2d_ws(d, x.cuda(), wt.cuda(), b.cuda(), al.cuda(), act, DT[dt], g.t,
                                gws.t, ws_bytes)
        assert st == 0, A.status_string(st)
        g.check(f"deconv tc {shape} act{act}")
        gws.check(f"deconv tc workspace {shape}")
        assert_parity(g.t, ref, TDT[dt], f"deconv tc {dt} {shape} act{act}")


# ---------------------------------------------------------------- frame prep
@pytest.mark.parametrize("hw", [(16, 24), (68, 120)])
@pytest.mark.parametrize("dt", ["f16", "f32"])
def test_frame_prep_quarter(hw, dt):
    h, w = hw
    f0 = G.rgba_frame(9, "f0", h, w)
    f1 = G.rgba_frame(9, "f1", h, w)
    g = Guarded((7, h // 4, w // 4), TDT[dt])
    y = A.frame_prep_quarter(f0.cuda(), f1.cuda(), 0.5, out_dtype=TDT[dt], out=g.t)
    g.check(f"prep {hw}")
    assert_parity(y, O.prep_quarter(f0.numpy(), f1.numpy(), 0.5), TDT[dt])


# ---------------------------------------------------------------- section runner
def test_section_graph_replay_matches_eager():
    x = G.tensor(10, "gx", (2, 12, 12, 64), "normal", dtype=G.BF16).cuda()
    wt = G.conv_weight(10, "g", 64, 64, 3, 3, G.NHWC, G.BF16).cuda()
    b = G.conv_bias(10, "g", 64).cuda()
    eager = A.pool2d(A.conv2d_fused(x, wt, b, pad=1, act=A.ACT_RELU), A.POOL_MAX, 3, 2, 1)
    s = torch.cuda.Stream()
    y1 = torch.empty(2, 12, 12, 64, dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty(2, 6, 6, 64, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        sec = A.Section(s)
        with sec:
            A.conv2d_fused(x, wt, b, pad=1, act=A.ACT_RELU, out=y1, stream=s)
            A.pool2d(y1, A.POOL_MAX, 3, 2, 1, out=y2, stream=s)
        y2.zero_()
        sec.launch()
        sec.launch()
    s.synchronize()
    assert torch.equal(y2, eager)
    sec.close()


# ---------------------------------------------------------------- split-K
SPLITK_CASES = [
    # name, n, h, w, cin, cout, k, s, p, layout, act, res
    ("s4_3x3", 8, 20, 20, 512, 512, 3, 1, 1, G.NHWC, A.ACT_RELU, A.RES_NONE),
    ("pan5_silu", 2, 20, 20, 512, 256, 3, 1, 1, G.NHWC, A.ACT_SILU, A.RES_NONE),
    ("res_prelu", 1, 17, 30, 240, 240, 3, 1, 1, G.NHWC, A.ACT_PRELU, A.RES_ACT_THEN_ADD),
    ("1x1_addres", 2, 10, 10, 2048, 256, 1, 1, 0, G.NHWC, A.ACT_RELU, A.RES_ADD_THEN_ACT),
]


def min_workspace(d, full):
    """Smallest workspace the call accepts (the NCHW staging copies; 0 for NHWC)."""
    if A.acnn_conv2d_plan(d, 0)[0] == 0:
        return 0
    lo, hi = 0, full
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if A.acnn_conv2d_plan(d, mid)[0] == 0:
            hi = mid
        else:
            lo = mid
    return hi


def test_conv_nchw_never_splits():
    """NCHW-output convs run unsplit (the plan query says so, and the workspace
    holds only the staging) even where the same NHWC conv splits K."""
    dn = A.ConvDesc(1, 17, 30, 240, 240, 3, 3, 1, 1, G.NCHW, G.F16)
    dh = A.ConvDesc(1, 17, 30, 240, 240, 3, 3, 1, 1, G.NHWC, G.F16)
    assert A.acnn_conv2d_plan(dh, A.acnn_conv2d_workspace_size(dh))[3] > 1
    st, _, _, sp = A.acnn_conv2d_plan(dn, A.acnn_conv2d_workspace_size(dn))
    assert st == 0 and sp == 1
    assert A.acnn_conv2d_workspace_size(dn) == A.acnn_conv2d_prepacked_workspace_size(dn) + \
        (240 * 9 * 240 * 2 + 255) // 256 * 256


@pytest.mark.parametrize("case", SPLITK_CASES, ids=[c[0] for c in SPLITK_CASES])
def test_conv_split_k(case):
    """Shapes whose plan splits K (fp32 partial tiles, reduced by the last split of each
    tile inside the kernel) match the oracle, and a workspace too small for the split
    gives the same answer unsplit."""
    name, n, h, w, cin, cout, k, s, p, layout, act, res_mode = case
    dt = "bf16" if layout == G.NHWC else "f16"
    d = A.ConvDesc(n, h, w, cin, cout, k, k, s, p, layout, DT[dt])
    full = A.acnn_conv2d_workspace_size(d)
    st, rows, bn, splits = A.acnn_conv2d_plan(d, full)
    assert st == 0 and splits > 1, (rows, bn, splits)
    y, ref = conv_case("sk" + name, n, h, w, cin, cout, k, s, p, dt, layout=layout, act=act,
                       res_mode=res_mode)
    assert_parity(y, ref, TDT[dt], name)
    # only the NCHW staging part of the workspace: the plan falls back to one split
    seed = 11
    x = G.tensor(seed, "sk" + name + ".x", G.activation_shape(layout, n, cin, h, w), "normal",
                 dtype=DT[dt]).cuda()
    wt = G.conv_weight(seed, "sk" + name, cout, cin, k, k, layout, DT[dt]).cuda()
    b = G.conv_bias(seed, "sk" + name, cout).cuda()
    al = G.prelu_alpha(seed, "sk" + name, cout).cuda()
    r = None
    if res_mode:
        oh, ow = (h + 2 * p - k) // s + 1, (w + 2 * p - k) // s + 1
        r = G.tensor(seed, "sk" + name + ".r", G.activation_shape(layout, n, cout, oh, ow),
                     "normal", dtype=DT[dt]).cuda()
    staging = min_workspace(d, full)
    st, _, _, sp1 = A.acnn_conv2d_plan(d, staging)
    assert st == 0 and sp1 == 1
    ws = torch.empty(max(staging, 16), dtype=torch.uint8, device="cuda")
    y1 = torch.empty_like(y)
    st = A.acnn_conv2d_fused(d, x, wt, b, al, r, res_mode, act, y1, ws if staging else None,
                             staging)
    assert st == 0, A.status_string(st)
    torch.cuda.synchronize()
    assert_parity(y1, ref, TDT[dt], name + " unsplit")
    # split twice through one workspace: the tile counters start from zero each
    # time and the split-order sum makes the result bitwise repeatable
    wsf = torch.empty(full, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        yk = torch.empty_like(y)
        st = A.acnn_conv2d_fused(d, x, wt, b, al, r, res_mode, act, yk, wsf, full)
        assert st == 0, A.status_string(st)
        outs.append(yk)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]), name + " split result not repeatable"
    assert_parity(outs[0], ref, TDT[dt], name + " reused workspace")


# ---------------------------------------------------------------- 256-row tiles
ROWS256_CASES = [
    # name, n, h, w, cin, cout, k, s, p, layout, act, res
    ("3x3_64", 4, 100, 100, 64, 64, 3, 1, 1, G.NHWC, A.ACT_RELU, A.RES_NONE),
    ("3x3_32_res", 4, 96, 100, 32, 32, 3, 1, 1, G.NHWC, A.ACT_SILU, A.RES_ACT_THEN_ADD),
    ("3x3_128_nchw", 2, 90, 120, 128, 128, 3, 1, 1, G.NCHW, A.ACT_PRELU, A.RES_ADD_THEN_ACT),
]


@pytest.mark.parametrize("case", ROWS256_CASES, ids=[c[0] for c in ROWS256_CASES])
def test_conv_256_row_tiles(case):
    """Narrow-output convs whose plan uses 256-pixel tiles (two 128-row MMAs per k-block)."""
    name, n, h, w, cin, cout, k, s, p, layout, act, res_mode = case
    dt = "bf16" if layout == G.NHWC else "f16"
    d = A.ConvDesc(n, h, w, cin, cout, k, k, s, p, layout, DT[dt])
    st, rows, bn, splits = A.acnn_conv2d_plan(d, A.acnn_conv2d_workspace_size(d))
    assert st == 0 and rows == 256, (rows, bn, splits)
    y, ref = conv_case("r256" + name, n, h, w, cin, cout, k, s, p, dt, layout=layout, act=act,
                       res_mode=res_mode)
    assert_parity(y, ref, TDT[dt], name)


# ---------------------------------------------------------------- flow out (NEXT-1)
def _flow_inputs(h, w, dt, seed=21, flow=3.0, mask_std=3.0):
    """Flows uniform in [-flow, flow] at 1/8 resolution (x8 on the page: up to
    8*flow pixels), mask logits N(0, mask_std), two random RGBA8 frames."""
    t = torch.cat([G.tensor(seed, "flow.uv", (4, h // 8, w // 8), "uniform", -flow, flow),
                   G.tensor(seed, "flow.mask", (1, h // 8, w // 8), "normal", std=mask_std)])
    t = t.to(TDT[dt])
    f0 = G.rgba_frame(seed, "flow.f0", h, w)
    f1 = G.rgba_frame(seed, "flow.f1", h, w)
    return t, f0, f1


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("hw", [(8, 8), (64, 96), (136, 200), (1088, 1920)])
def test_flow_out_bytes(dt, hw):
    """Every output byte equals the binary32 oracle's (same operation order,
    no fused multiply-adds), except a difference of one where the oracle's
    pre-byte value lies at a byte boundary: the two sides take the mask's exp
    from different libraries (CUDA's expf, the C library's exp)."""
    h, w = hw
    t, f0, f1 = _flow_inputs(h, w, dt)
    g = Guarded((h, w, 4), torch.uint8)
    y = A.frame_flow_out(t.cuda(), f0.cuda(), f1.cuda(), out=g.t)
    g.check(f"flow_out {hw}")
    ref, pre = O.flow_out(t.float().numpy(), f0.numpy(), f1.numpy(), with_pre=True)
    assert_bytes_boundary(y, ref, pre, f"flow_out {dt} {hw}")


@pytest.mark.parametrize("flow,mask_std", [(200.0, 40.0), (0.0, 0.0), (0.125, 100.0)])
def test_flow_out_extremes(flow, mask_std):
    """Flows far outside the frame (clamped taps), zero flow and mask 0 (m = 1/2,
    exact on both sides: bit-exact), whole-pixel flows with saturated masks."""
    h, w = 72, 136
    t, f0, f1 = _flow_inputs(h, w, "f32", seed=22, flow=flow, mask_std=mask_std)
    y = A.frame_flow_out(t.cuda(), f0.cuda(), f1.cuda())
    torch.cuda.synchronize()
    ref, pre = O.flow_out(t.numpy(), f0.numpy(), f1.numpy(), with_pre=True)
    n1 = assert_bytes_boundary(y, ref, pre, f"flow_out extremes {flow} {mask_std}")
    if mask_std == 0.0:
        assert n1 == 0


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("hw", [(8, 8), (64, 96), (1088, 1920)])
def test_flow_out_refine_residual(dt, hw):
    """With the refine residual (x4 bilinear upsample added before the clamp),
    the bytes still follow the binary32 oracle's under the boundary rule."""
    h, w = hw
    t, f0, f1 = _flow_inputs(h, w, dt, seed=23)
    res = G.tensor(23, "flow.res", (3, h // 4, w // 4), "uniform", -0.4, 0.4)
    y = A.frame_flow_out(t.cuda(), f0.cuda(), f1.cuda(), refine_res=res.cuda())
    torch.cuda.synchronize()
    ref, pre = O.flow_out(t.float().numpy(), f0.numpy(), f1.numpy(), res=res.numpy(),
                          with_pre=True)
    assert_bytes_boundary(y, ref, pre, f"flow_out+res {dt} {hw}")
    # a residual moves bytes: the frame differs from the one without it
    y0 = A.frame_flow_out(t.cuda(), f0.cuda(), f1.cuda())
    assert not torch.equal(y0, y)


# ---------------------------------------------------------------- t-factored stack (NEXT-3)
def _prep_bound(h, w, flow):
    """Refine prep in fp32 against the fp64 oracle.  Every value is a bilinear
    (continuous, slope <= 1 per pixel for [0, 1] planes) function of tap
    positions that fp32 carries with an absolute error of a few ulp of the
    largest coordinate (max(h, w) + 8 * flow pixels); the flow planes are
    scaled down by 80.  So 8 ulp of that coordinate, plus fp32 rounding of
    the results themselves, bounds the difference."""
    return 8 * (max(h, w) + 8 * flow) * 2.0 ** -24 + 1e-6


@pytest.mark.parametrize("dt,out", [("f32", "f32"), ("f16", "f16"), ("bf16", "bf16"),
                                    ("f16", "f32")])
@pytest.mark.parametrize("hw", [(8, 8), (64, 96), (136, 200)])
def test_refine_prep(dt, out, hw):
    h, w = hw
    t, f0, f1 = _flow_inputs(h, w, dt, seed=24)
    g = Guarded((11, h // 4, w // 4), TDT[out])
    y = A.frame_refine_prep(t.cuda(), f0.cuda(), f1.cuda(), out_dtype=TDT[out], out=g.t)
    g.check(f"refine_prep {hw}")
    ref = O.refine_prep(t.double().numpy(), f0.numpy(), f1.numpy())
    assert tuple(y.shape) == (11, h // 4, w // 4)
    if out == "f32":
        err = np.abs(to64(y) - ref).max()
        assert err <= _prep_bound(h, w, 3.0), (hw, err)
    else:
        assert_parity(y, ref, TDT[out], f"refine_prep {dt}->{out} {hw}")


def test_refine_prep_full_size():
    """1088x1920 (the workload's size), fp16 in and out, on every value."""
    h, w = 1088, 1920
    t, f0, f1 = _flow_inputs(h, w, "f16", seed=25)
    y = A.frame_refine_prep(t.cuda(), f0.cuda(), f1.cuda(), out_dtype=torch.float16)
    torch.cuda.synchronize()
    ref = O.refine_prep(t.double().numpy(), f0.numpy(), f1.numpy())
    assert_parity(y, ref, torch.float16, "refine_prep full")
    y32 = A.frame_refine_prep(t.cuda(), f0.cuda(), f1.cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    err = np.abs(to64(y32) - ref).max()
    assert err <= _prep_bound(h, w, 3.0), err


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("c,hh,hw", [(32, 272, 480), (11, 7, 9), (70, 33, 65), (1, 1, 1),
                                     (4, 1, 37), (64, 40, 1)])
def test_refine_out(dt, c, hh, hw):
    """Replicate-padded 3x3 C -> 3, fp32 accumulation and output; sizes off the
    32x8 block, a channel count across the 64-channel weight chunks, 1-pixel
    rows and columns where every tap clamps."""
    x = G.tensor(26, f"ro.x{c}", (c, hh, hw), "normal", dtype=DT[dt])
    wt = G.conv_weight(26, f"ro{c}", 3, c, 3, 3, G.NCHW, G.F32)
    b = G.conv_bias(26, f"ro{c}", 3)
    g = Guarded((3, hh, hw), torch.float32)
    y = A.frame_refine_out(x.cuda(), wt.cuda(), b.cuda(), out=g.t)
    g.check(f"refine_out {c}x{hh}x{hw}")
    ref = O.refine_out(to64(x), to64(wt), to64(b))
    assert_parity(y, ref, torch.float32, f"refine_out {dt} {c}x{hh}x{hw}")


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("t", [0.0, 0.5, 1.0])
@pytest.mark.parametrize("c,n,hn", [(240, 68 * 120, 64), (3, 1, 1), (17, 1000, 5)])
def test_film(dt, t, c, n, hn):
    x = G.tensor(27, f"film.x{c}", (c, n), "normal", dtype=DT[dt])
    prm = G.film_mlp(27, f"film{c}", c, hn)
    g = Guarded(x.shape, TDT[dt])
    y = A.film(x.cuda(), t, *[p.cuda() for p in prm], out=g.t)
    g.check(f"film {c}x{n}")
    ref = O.film(to64(x), t, *[to64(p) for p in prm])
    assert_parity(y, ref, TDT[dt], f"film {dt} t={t} {c}x{n}")


def test_film_in_place():
    c, n = 64, 4096
    x = G.tensor(28, "film.xi", (c, n), "normal", dtype=G.F16).cuda()
    prm = [p.cuda() for p in G.film_mlp(28, "filmi", c, 32)]
    y = A.film(x, 0.3, *prm)
    A.film(x, 0.3, *prm, out=x)
    torch.cuda.synchronize()
    assert torch.equal(x, y)


# ---------------------------------------------------------------- concat folded into the conv (NEXT-2)
CAT_CASES = [
    # name, n, h, w, c_a, c_b, cout, k, s, p, act, res
    ("neck_3x3", 2, 20, 20, 256, 256, 256, 3, 1, 1, A.ACT_SILU, A.RES_NONE),
    ("1x1_res", 2, 12, 17, 64, 128, 128, 1, 1, 0, A.ACT_RELU, A.RES_ADD_THEN_ACT),
    ("3x3_s2_prelu", 1, 23, 19, 128, 64, 96, 3, 2, 1, A.ACT_PRELU, A.RES_NONE),
    ("big_m", 4, 40, 40, 256, 256, 256, 3, 1, 1, A.ACT_SILU, A.RES_NONE),
]


@pytest.mark.parametrize("case", CAT_CASES, ids=[c[0] for c in CAT_CASES])
def test_conv_cat2(case):
    """conv over [x_a | x_b] matches the oracle's concat + conv, and equals the
    library's own concat + conv2d_fused bit for bit."""
    name, n, h, w, ca, cb, cout, k, s, p, act, res_mode = case
    seed = 31
    xa = G.tensor(seed, name + ".xa", (n, h, w, ca), "normal", dtype=G.BF16)
    xb = G.tensor(seed, name + ".xb", (n, h, w, cb), "normal", dtype=G.BF16)
    wt = G.conv_weight(seed, name, cout, ca + cb, k, k, G.NHWC, G.BF16)
    b = G.conv_bias(seed, name, cout)
    al = G.prelu_alpha(seed, name, cout)
    oh, ow = (h + 2 * p - k) // s + 1, (w + 2 * p - k) // s + 1
    r = G.tensor(seed, name + ".r", (n, oh, ow, cout), "normal", dtype=G.BF16) if res_mode else None
    dev = lambda t: None if t is None else t.cuda()
    y = A.conv2d_fused_cat2(dev(xa), dev(xb), dev(wt), dev(b), stride=s, pad=p, act=act,
                            alpha=dev(al), residual=dev(r), res_mode=res_mode)
    cat = A.concat(dev(xa), dev(xb))
    y2 = A.conv2d_fused(cat, dev(wt), dev(b), stride=s, pad=p, act=act, alpha=dev(al),
                        residual=dev(r), res_mode=res_mode)
    torch.cuda.synchronize()
    assert torch.equal(y, y2), name + ": folded concat differs from concat + conv"
    ref = O.conv2d(O.concat(to64(xa), to64(xb)), to64(wt), to64(b), stride=s, pad=p, act=act,
                   alpha=to64(al), residual=None if r is None else to64(r), res_mode=res_mode)
    assert_parity(y, ref, torch.bfloat16, name)
