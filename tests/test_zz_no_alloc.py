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
from tests.parity import assert_parity, to64


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
        assert_parity(y_na, to64(y_ref), torch.float16, f"call {call} vs workspace entry")
        ref = O.conv2d(to64(x), to64(wt), to64(b), pad=1, act=O.ACT_PRELU, alpha=to64(al),
                       residual=to64(r), res_mode=O.RES_ACT_THEN_ADD, layout=O.NCHW)
        assert_parity(y_na, ref, torch.float16, f"call {call} vs oracle")
    assert A.acnn_last_device_status() == 0
