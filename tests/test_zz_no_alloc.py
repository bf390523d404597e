"""acnn_conv2d_fused_noalloc: the conv entry point for callers that cannot allocate.

Callers such as a plugin running inside a framework that owns all device
memory (and hands the plugin no allocator), or a latency-critical loop where a
cudaMalloc could synchronise the device, cannot supply the workspace that the
NCHW tensor-core path needs.  The no-allocation entry point takes that scratch
from a static device array in the library instead.  These tests call it through
the C ABI and check it against the ordinary entry point (and the oracle) on two
calls in a row, so that a stale or shared scratch would show.  This file is
collected last on purpose.
"""
import pytest
import torch

from activation_cnn_gb300 import acnn as A
from activation_cnn_gb300 import inputs as G
from oracle import oracle as O
from tests.parity import assert_bitexact, assert_parity, to64


def test_noalloc_rejects_oversized_scratch():
    """A geometry needing more scratch than the static array: clear error, no launch."""
    d = A.ConvDesc(1, 256, 256, 256, 256, 3, 3, 1, 1, G.NCHW, G.F16)
    assert A.acnn_conv2d_workspace_size(d) > A.NOALLOC_SCRATCH_BYTES
    X, W, Y = 0x1000000, 0x9000000, 0x11000000  # never dereferenced
    st = A.acnn_conv2d_fused_noalloc(d, X, W, None, None, None, 0, 0, Y, 0)
    assert st == 5, A.status_string(st)  # ACNN_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from activation_cnn_gb300 import build
    build.build()
    A.lib()
    n, c_in, c_out, h, w = 1, 120, 240, 36, 62
    d = A.ConvDesc(n, h, w, c_in, c_out, 3, 3, 1, 1, G.NCHW, G.F16)
    need = A.acnn_conv2d_workspace_size(d)
    assert 0 < need <= A.NOALLOC_SCRATCH_BYTES
    wt = G.conv_weight(21, "na", c_out, c_in, 3, 3, G.NCHW, G.F16)
    b = G.conv_bias(21, "na", c_out)
    al = G.prelu_alpha(21, "na", c_out)
    wd, bd, ald = wt.cuda(), b.cuda(), al.cuda()
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for call in range(2):  # two calls in a row: the shared scratch must not leak between them
        x = G.tensor(21, f"na.x{call}", (n, c_in, h, w), "normal", dtype=G.F16)
        r = G.tensor(21, f"na.r{call}", (n, c_out, h, w), "normal", dtype=G.F16)
        xd, rd = x.cuda(), r.cuda()
        y_ref = torch.empty((n, c_out, h, w), dtype=torch.float16, device="cuda")
        y_na = torch.full((n, c_out, h, w), float("nan"), dtype=torch.float16, device="cuda")
        st = A.acnn_conv2d_fused(d, xd, wd, bd, ald, rd, A.RES_ACT_THEN_ADD, A.ACT_PRELU, y_ref,
                                 ws, need)
        assert st == 0, A.status_string(st)
        st = A.acnn_conv2d_fused_noalloc(d, xd, wd, bd, ald, rd, A.RES_ACT_THEN_ADD,
                                         A.ACT_PRELU, y_na)
        assert st == 0, A.status_string(st)
        torch.cuda.synchronize()
        # same path, same plan, same staging layout: the same bits
        assert_bitexact(y_na, y_ref, f"call {call} vs workspace entry")
        ref = O.conv2d(to64(x), to64(wt), to64(b), pad=1, act=O.ACT_PRELU, alpha=to64(al),
                       residual=to64(r), res_mode=O.RES_ACT_THEN_ADD, layout=O.NCHW)
        assert_parity(y_na, ref, torch.float16, f"call {call} vs oracle")
    assert A.acnn_last_device_status() == 0


@pytest.mark.gpu
def test_noalloc_nhwc_split_k_beyond_the_array_twice():
    """An NHWC bf16 conv whose full split-K workspace is larger than the static
    array (it needs no staging): the entry point plans fewer splits into the
    array.  Two calls in a row give the same bits, the same bits as the
    workspace entry point given a workspace of the array's size (the same
    plan), and match the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from activation_cnn_gb300 import build
    build.build()
    A.lib()
    cands = [(8, 20, 20, 512, 512), (8, 40, 40, 256, 256), (16, 20, 20, 512, 512),
             (8, 20, 20, 1024, 1024)]
    pick = None
    for n, h, w, ci, co in cands:
        d = A.ConvDesc(n, h, w, ci, co, 3, 3, 1, 1, G.NHWC, G.BF16)
        if A.acnn_conv2d_workspace_size(d) > A.NOALLOC_SCRATCH_BYTES:
            pick = (n, h, w, ci, co, d)
            break
    assert pick is not None, "no candidate splits K beyond the static array"
    n, h, w, ci, co, d = pick
    st, _, _, splits = A.acnn_conv2d_plan(d, A.NOALLOC_SCRATCH_BYTES)
    assert st == 0
    print(f"geometry {pick[:5]}: {splits} splits within the array")
    x = G.tensor(22, "nah.x", (n, h, w, ci), "normal", dtype=G.BF16)
    wt = G.conv_weight(22, "nah", co, ci, 3, 3, G.NHWC, G.BF16)
    b = G.conv_bias(22, "nah", co)
    xd, wd, bd = x.cuda(), wt.cuda(), b.cuda()
    ws = torch.empty(A.NOALLOC_SCRATCH_BYTES, dtype=torch.uint8, device="cuda")
    y_ref = torch.empty((n, h, w, co), dtype=torch.bfloat16, device="cuda")
    st = A.acnn_conv2d_fused(d, xd, wd, bd, None, None, A.RES_NONE, A.ACT_RELU, y_ref, ws,
                             A.NOALLOC_SCRATCH_BYTES)
    assert st == 0, A.status_string(st)
    ref = O.conv2d(to64(x), to64(wt), to64(b), pad=1, act=O.ACT_RELU)
    outs = []
    for call in range(2):
        y_na = torch.full((n, h, w, co), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = A.acnn_conv2d_fused_noalloc(d, xd, wd, bd, None, None, A.RES_NONE, A.ACT_RELU, y_na)
        assert st == 0, A.status_string(st)
        torch.cuda.synchronize()
        assert_bitexact(y_na, y_ref, f"call {call} vs workspace entry")
        assert_parity(y_na, ref, torch.bfloat16, f"call {call} vs oracle")
        outs.append(y_na)
    assert torch.equal(outs[0], outs[1])
    assert A.acnn_last_device_status() == 0
