"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before any CUDA call."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def A():
    from activation_cnn_gb300 import build
    build.build()
    from activation_cnn_gb300 import acnn
    acnn.lib()
    return acnn


def declared_symbols():
    with open(os.path.join(ROOT, "include", "acnn.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(acnn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_binding_names():
    from activation_cnn_gb300 import acnn
    assert sorted(acnn.EXPORTS) == declared_symbols()


def test_library_exports_every_declared_symbol(A):
    lib = A.lib()
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing


def test_status_strings(A):
    for code in range(11):
        assert A.status_string(code) and A.status_string(code) != "unknown status"
    assert A.status_string(999) == "unknown status"


def desc(A, **kw):
    d = dict(n=1, h=8, w=8, c_in=16, c_out=32, kh=3, kw=3, stride=1, pad=1, layout=0, dtype=2)
    d.update(kw)
    return A.ConvDesc(*[d[k] for k in ("n", "h", "w", "c_in", "c_out", "kh", "kw", "stride",
                                       "pad", "layout", "dtype")])


X, W, Y, R, B = 0x1000000, 0x2000000, 0x3000000, 0x4000000, 0x5000000  # never dereferenced


def test_conv_rejects_before_launch(A):
    c = A.acnn_conv2d_fused
    d = desc(A)
    assert c(d, None, W, None, None, None, 0, 0, Y, None, 0, 0) == 1          # NULL x
    assert c(d, X, W, None, None, None, 0, A.ACT_PRELU, Y, None, 0, 0) == 1   # PReLU w/o alpha
    assert c(d, X, W, None, None, None, 1, 0, Y, None, 0, 0) == 1             # residual missing
    assert c(d, X, W, None, None, None, 0, 9, Y, None, 0, 0) == 7             # bad act
    assert c(d, X, W, None, None, None, 5, 0, Y, None, 0, 0) == 7             # bad res mode
    assert c(desc(A, dtype=5), X, W, None, None, None, 0, 0, Y, None, 0, 0) == 7
    assert c(desc(A, layout=3), X, W, None, None, None, 0, 0, Y, None, 0, 0) == 7
    assert c(desc(A, n=0), X, W, None, None, None, 0, 0, Y, None, 0, 0) == 2
    assert c(desc(A, h=1, pad=0), X, W, None, None, None, 0, 0, Y, None, 0, 0) == 2
    assert c(desc(A, stride=0), X, W, None, None, None, 0, 0, Y, None, 0, 0) == 2
    assert c(d, X + 4, W, None, None, None, 0, 0, Y, None, 0, 0) == 4        # misaligned
    assert c(d, X, W, B + 4, None, None, 0, 0, Y, None, 0, 0) == 4
    assert c(d, X, W, None, None, None, 0, 0, X + 256, None, 0, 0) == 6      # y overlaps x
    # NCHW on the tensor path needs its workspace
    dn = desc(A, layout=1, c_in=64, c_out=64)
    assert A.acnn_conv2d_workspace_size(dn) > 0
    assert c(dn, X, W, None, None, None, 0, 0, Y, None, 0, 0) == 5


def test_conv_path_selection(A):
    assert A.acnn_conv2d_path(desc(A, c_in=64, c_out=64, kh=1, kw=1, pad=0)) == 1
    assert A.acnn_conv2d_path(desc(A, c_in=64, c_out=64)) == 2
    assert A.acnn_conv2d_path(desc(A, c_in=64, c_out=64, stride=2)) == 2
    assert A.acnn_conv2d_path(desc(A, c_in=3, c_out=32)) == 3         # tiny C_in: packed
    assert A.acnn_conv2d_path(desc(A, c_in=7, c_out=120, layout=1, dtype=1)) == 3
    assert A.acnn_conv2d_path(desc(A, c_in=5, c_out=32)) == 3
    assert A.acnn_conv2d_path(desc(A, c_in=3, c_out=32, dtype=0)) == 0  # fp32: FFMA direct
    assert A.acnn_conv2d_path(desc(A, dtype=0)) == 0                  # fp32
    assert A.acnn_conv2d_path(desc(A, c_in=64, c_out=120)) == 2       # C_out % 8 == 0
    assert A.acnn_conv2d_path(desc(A, c_in=64, c_out=30)) == 0        # C_out % 8 != 0
    assert A.acnn_conv2d_path(desc(A, c_in=8, c_out=64, kw=1, pad=0)) == 3  # non-square
    assert A.acnn_conv2d_path(desc(A, c_in=64, c_out=64, kw=1, pad=0)) == 3
    assert A.acnn_conv2d_path(desc(A, c_in=100, c_out=64, kh=3, kw=3)) == 0  # K > 512
    assert A.acnn_conv2d_path(desc(A, c_in=64, c_out=4096)) == 2
    assert A.acnn_conv2d_path(desc(A, c_in=64, c_out=4104)) == 0      # C_out > 4096
    # beyond the packed path's C_out limit the tiny-C_in direct kernel serves
    assert A.acnn_conv2d_path(desc(A, c_in=3, c_out=4104)) == 4
    assert A.acnn_conv2d_path(desc(A, c_in=5, c_out=4104)) == 0
    assert A.acnn_conv2d_workspace_size(desc(A, c_in=3, c_out=4104)) == 0
    assert A.acnn_conv2d_workspace_size(desc(A, c_in=3, c_out=32)) >= 64 * 32 * 2
    assert A.acnn_conv2d_path(desc(A, n=0)) == -1
    assert A.acnn_conv2d_workspace_size(desc(A, c_in=64, c_out=64)) == 0


def test_conv_pool2_rejects_before_launch(A):
    """The conv with a pooled second output validates on the host: geometry it
    does not serve, a missing pooled buffer, misalignment and aliasing."""
    def c(*args):
        return A.acnn_conv2d_fused_pool2(*args, 0)  # stream 0: nothing is enqueued
    ok = desc(A, c_in=64, c_out=64, kh=1, kw=1, pad=0)
    P = 0x6000000
    assert c(desc(A, c_in=64, c_out=64), X, W, None, None, None, 0, 0, Y, P) == 3     # 3x3
    assert c(desc(A, c_in=64, c_out=64, kh=1, kw=1, pad=0, h=7), X, W, None, None, None, 0, 0,
             Y, P) == 3                                                              # odd height
    assert c(desc(A, c_in=32, c_out=64, kh=1, kw=1, pad=0), X, W, None, None, None, 0, 0,
             Y, P) == 3                                                              # C_in < 64
    assert c(desc(A, c_in=64, c_out=64, kh=1, kw=1, pad=0, layout=1), X, W, None, None, None,
             0, 0, Y, P) == 3                                                        # NCHW
    assert c(ok, X, W, None, None, None, 0, 0, Y, None) == 1                           # no y_pool
    assert c(ok, X, W, None, None, None, 0, 0, Y, P + 8) == 4                          # misaligned
    assert c(ok, X, W, None, None, None, 0, 0, Y, Y + 64) == 6                         # y_pool in y
    assert c(ok, X, W, None, None, None, 0, 0, Y, X) == 6                              # y_pool in x
    assert c(ok, X, W, None, None, None, 0, 9, Y, P) == 7                              # bad act


def test_conv_up2_rejects_before_launch(A):
    """The conv with an upsampled second output validates on the host."""
    def c(dsc, x_b, y_up, c_a=0, act=0):
        return A.acnn_conv2d_fused_up2(dsc, X, c_a, x_b, W, None, None, None, 0, act, Y, y_up,
                                       None, 0, 0)
    U = 0x7000000
    ok = desc(A, c_in=64, c_out=64)
    assert c(desc(A, c_in=64, c_out=64, layout=1, dtype=1), None, U) == 3     # NCHW
    assert c(desc(A, c_in=64, c_out=64, dtype=0), None, U) == 3               # fp32
    assert c(desc(A, c_in=128, c_out=64), R, U, c_a=32) == 3                  # c_a % 64
    assert c(ok, None, None) == 1                                             # no y_up
    assert c(ok, None, U + 8) == 4                                            # misaligned
    assert c(ok, None, Y + 64) == 6                                           # y_up in y
    assert c(ok, None, U, act=9) == 7


def test_deconv_tensor_core_workspace(A):
    """The tensor-core deconv's workspace: for fp16/bf16 with out = in dtype and
    c_in % 8 == 0 only (0 otherwise: the direct kernel serves)."""
    def d(**kw):
        return desc(A, **dict(dict(c_in=240, c_out=5, kh=4, kw=4, stride=2, pad=1, layout=1,
                                   dtype=1, h=68, w=120), **kw))
    es = 2
    co4 = 24
    want = (((68 * 120 * 240 * es + 255) // 256 * 256) + ((co4 * 9 * 240 * es + 255) // 256 * 256)
            + 2 * 256 + ((68 * 120 * co4 * es + 255) // 256 * 256))
    assert A.acnn_deconv2d_workspace_size(d(), 1) == want
    assert A.acnn_deconv2d_workspace_size(d(layout=0), 1) == want - (68 * 120 * 240 * es + 255) // 256 * 256
    assert A.acnn_deconv2d_workspace_size(d(), 0) == 0          # fp32 output
    assert A.acnn_deconv2d_workspace_size(d(dtype=0), 0) == 0   # fp32 input
    assert A.acnn_deconv2d_workspace_size(d(c_in=20), 1) == 0   # c_in % 8
    assert A.acnn_deconv2d_workspace_size(d(dtype=2), 2) == 0   # bf16: the direct kernel
    assert A.acnn_deconv2d_workspace_size(d(stride=1), 1) == 0


def test_force_path_selects_the_tiny_kernel(A):
    """The tuning hook routes the 3/6/7-channel 3x3 convs to the direct kernel
    (and nothing else), and path 0 restores the router."""
    try:
        assert A.acnn_conv2d_force_path(4, 1) == 0
        assert A.acnn_conv2d_path(desc(A, c_in=3, c_out=32)) == 4
        assert A.acnn_conv2d_path(desc(A, c_in=6, c_out=120, layout=1, dtype=1)) == 4
        assert A.acnn_conv2d_workspace_size(desc(A, c_in=7, c_out=120, layout=1, dtype=1)) == 0
        assert A.acnn_conv2d_path(desc(A, c_in=5, c_out=32)) == 3      # not a tiny geometry
        assert A.acnn_conv2d_path(desc(A, c_in=3, c_out=32, stride=3)) == 3
        assert A.acnn_conv2d_path(desc(A, c_in=3, c_out=32, dtype=0)) == 0
    finally:
        assert A.acnn_conv2d_force_path(0, 0) == 0
    assert A.acnn_conv2d_path(desc(A, c_in=3, c_out=32)) == 3
    assert A.acnn_conv2d_force_path(2, 0) == 7 and A.acnn_conv2d_force_path(4, 2) == 7


def test_conv_out_hw(A):
    st, oh, ow = A.acnn_conv2d_out_hw(desc(A, h=640, w=640, stride=2))
    assert (st, oh, ow) == (0, 320, 320)
    st, oh, ow = A.acnn_conv2d_out_hw(desc(A, h=7, w=9, kh=3, kw=3, stride=2, pad=1))
    assert (st, oh, ow) == (0, 4, 5)


def test_companions_reject_before_launch(A):
    assert A.acnn_pool2d(2, 1, 8, 8, 4, 3, 2, 1, 0, 0, X, Y, 0) == 7           # bad kind
    assert A.acnn_pool2d(1, 1, 8, 8, 4, 2, 2, 1, 0, 0, X, Y, 0) == 3           # avg with pad
    assert A.acnn_pool2d(0, 1, 8, 8, 4, 3, 2, 3, 0, 0, X, Y, 0) == 3           # pad >= k
    assert A.acnn_pool2d(0, 1, 8, 8, 4, 3, 2, 1, 0, 0, None, Y, 0) == 1
    assert A.acnn_pool2d(0, 1, 8, 8, 4, 3, 2, 1, 0, 0, X, X + 16, 0) == 6
    assert A.acnn_resize2d(0, 1, 4, 8, 8, 16, 16, 0, 2, 0, X, Y, 0) == 3       # nearest casts
    assert A.acnn_resize2d(1, 1, 4, 8, 8, 0, 16, 0, 2, 2, X, Y, 0) == 2
    assert A.acnn_resize2d(3, 1, 4, 8, 8, 4, 16, 0, 2, 2, X, Y, 0) == 7
    assert A.acnn_concat(1, 4, 4, 8, 8, 0, 2, X, W, X + 32, 0) == 6
    assert A.acnn_concat(1, 4, 4, 0, 8, 0, 2, X, W, Y, 0) == 2
    d = desc(A, kh=3, kw=3, stride=2, pad=1)
    assert A.acnn_deconv2d(d, X, W, None, None, 0, 1, Y, 0) == 3               # only 4/2/1
    d4 = desc(A, kh=4, kw=4, stride=2, pad=1)
    assert A.acnn_deconv2d(d4, X, W, None, None, 0, 7, Y, 0) == 7
    assert A.acnn_frame_prep_quarter(10, 16, X, W, 0.5, 1, Y, 0) == 2          # h % 4
    assert A.acnn_frame_prep_quarter(16, 16, X, None, 0.5, 1, Y, 0) == 1
    # flow out: h, w multiples of 8, dtype enum, pointers, alignment, aliasing
    assert A.acnn_frame_flow_out(12, 16, X, 1, W, Y, None, Y + (1 << 20), 0) == 2
    assert A.acnn_frame_flow_out(16, 16, X, 9, W, Y, None, Y + (1 << 20), 0) == 7
    assert A.acnn_frame_flow_out(16, 16, None, 1, W, Y, None, Y + (1 << 20), 0) == 1
    assert A.acnn_frame_flow_out(16, 16, X, 1, W + 4, Y, None, Y + (1 << 20), 0) == 4
    assert A.acnn_frame_flow_out(16, 16, X, 1, W, Y, None, W + 512, 0) == 6
    assert A.acnn_frame_flow_out(16, 16, X, 1, W, Y, R + 4, Y + (1 << 20), 0) == 4  # residual
    assert A.acnn_frame_flow_out(16, 16, X, 1, W, Y, Y + (1 << 20), Y + (1 << 20), 0) == 6
    # prepacked weights: pointers, alignment, aliasing, geometry
    d3 = desc(A, kh=3, kw=3, stride=1, pad=1)
    assert A.acnn_conv2d_prepack(d3, None, Y, 0) == 1
    assert A.acnn_conv2d_prepack(d3, W, W + 16, 0) == 6
    assert A.acnn_conv2d_prepack(d3, W + 4, Y, 0) == 4
    bad = desc(A, kh=3, kw=3, stride=0, pad=1)
    assert A.acnn_conv2d_prepack(bad, W, Y, 0) != 0
    assert A.acnn_conv2d_prepacked_size(bad) == 0
    assert A.acnn_conv2d_fused_prepacked(d3, X, None, None, None, None, 0, 1, Y, None, 0, 0) == 1
    assert A.acnn_conv2d_fused_prepacked(d3, X, W, None, None, None, 0, 9, Y, None, 0, 0) == 7
    # t-factored stack: refine prep / refine out / FiLM argument checks
    assert A.acnn_frame_refine_prep(12, 16, X, 1, W, Y, 1, R, 0) == 2
    assert A.acnn_frame_refine_prep(16, 16, X, 1, W, Y, 5, R, 0) == 7
    assert A.acnn_frame_refine_prep(16, 16, X, 1, None, Y, 1, R, 0) == 1
    assert A.acnn_frame_refine_prep(16, 16, X, 1, W, Y, 1, W + 64, 0) == 6
    assert A.acnn_frame_refine_out(0, 4, 4, X, 1, W, W + 512, R, 0) == 2
    assert A.acnn_frame_refine_out(8, 4, 4, X, 1, W, None, R, 0) == 1
    assert A.acnn_frame_refine_out(8, 4, 4, X, 1, W, W + 512, X + 16, 0) == 6
    assert A.acnn_frame_refine_out(8, 4, 4, X + 4, 1, W, W + 512, R, 0) == 4
    assert A.acnn_film(8, 16, 1, X, 0.5, W, W, 4, W, W, X, 0) != 6              # in place ok
    assert A.acnn_film(8, 16, 1, X, 0.5, W, W, 4, W, W, X + 2, 0) == 6
    assert A.acnn_film(8, 16, 1, X, 0.5, W, W, 0, W, W, Y, 0) == 2
    assert A.acnn_film(8, 16, 1, X, 0.5, W, None, 4, W, W, Y, 0) == 1
    assert A.acnn_film(70000, 16, 1, X, 0.5, W, W, 4, W, W, Y, 0) == 10         # c > 65535
    # folded concat conv: NHWC fp16/bf16 only, c_a a multiple of 64, c_b > 0
    d = desc(A, c_in=128, c_out=64)
    assert A.acnn_conv2d_fused_cat2(d, X, 64, R, W, None, None, None, 0, 1, Y, None, 0, 0) != 1
    assert A.acnn_conv2d_fused_cat2(d, X, 32, R, W, None, None, None, 0, 1, Y, None, 0, 0) == 3
    assert A.acnn_conv2d_fused_cat2(d, X, 128, R, W, None, None, None, 0, 1, Y, None, 0, 0) == 3
    assert A.acnn_conv2d_fused_cat2(d, X, 64, None, W, None, None, None, 0, 1, Y, None, 0, 0) == 1
    dn = desc(A, c_in=128, c_out=64, layout=1)
    assert A.acnn_conv2d_fused_cat2(dn, X, 64, R, W, None, None, None, 0, 1, Y, None, 0, 0) == 3
    assert A.acnn_conv2d_fused_cat2(d, X, 64, R, W, None, None, None, 0, 1, X + 64, None, 0,
                                    0) == 6


def test_wait_budget_knob(A):
    assert A.acnn_set_wait_budget(-1) == 2
    assert A.acnn_set_wait_budget(0) == 0


def test_section_end_null(A):
    assert A.lib().acnn_section_end(None, None) == 1
    assert A.acnn_section_launch(None, 0) == 1
    assert A.acnn_section_destroy(None) == 0


def test_per_device_opt_in_bookkeeping(tmp_path):
    """The per-device record behind the dynamic shared-memory opt-in
    (csrc/per_device.h), compiled on the host with g++: a kernel opted in on
    one device is not taken as opted in on another, larger requests are
    applied again, failures are not recorded, concurrent callers apply once."""
    import shutil
    import subprocess
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    exe = str(tmp_path / "per_device_check")
    subprocess.run([gxx, "-std=c++17", "-O1", "-pthread",
                    "-I", os.path.join(root, "activation_cnn_gb300", "csrc"),
                    os.path.join(root, "tests", "per_device_check.cpp"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
