"""Device-side failure detection without a GPU fault.

Every pipeline wait of the tensor-core conv is bounded.  With the debug knob
acnn_set_wait_budget(1) a wait gives up after one poll: the kernel records
ACNN_ERR_DEVICE_TIMEOUT in its status word, drains the copies and MMAs it
started, frees its tensor memory and returns -- no trap, no hang.  The host
reads the status with acnn_last_device_status; the context stays usable and
the next call (budget restored) is correct.
"""
import pytest
import torch

from activation_cnn_gb300 import acnn as A
from activation_cnn_gb300 import inputs as G
from oracle import oracle as O
from tests.parity import assert_parity, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _restore_budget():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from activation_cnn_gb300 import build
    build.build()
    yield
    A.acnn_set_wait_budget(0)


def test_expired_waits_report_timeout_and_context_survives():
    n, h, w, cin, cout = 2, 24, 24, 256, 256
    x = G.tensor(31, "fx", (n, h, w, cin), "normal", dtype=G.BF16)
    wt = G.conv_weight(31, "fw", cout, cin, 3, 3, G.NHWC, G.BF16)
    b = G.conv_bias(31, "fw", cout)
    xd, wd, bd = x.cuda(), wt.cuda(), b.cuda()
    y = torch.empty((n, h, w, cout), dtype=torch.bfloat16, device="cuda")
    d = A.ConvDesc(n, h, w, cin, cout, 3, 3, 1, 1, G.NHWC, G.BF16)
    ws = torch.empty(max(A.acnn_conv2d_workspace_size(d), 16), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    assert A.acnn_last_device_status() == 0

    assert A.acnn_set_wait_budget(1) == 0
    st = A.acnn_conv2d_fused(d, xd, wd, bd, None, None, A.RES_NONE, A.ACT_RELU, y, ws,
                             ws.numel())
    assert st == 0, A.status_string(st)   # the launch itself is valid
    assert A.acnn_last_device_status() == 9  # ACNN_ERR_DEVICE_TIMEOUT, read and cleared
    assert A.acnn_last_device_status() == 0

    A.acnn_set_wait_budget(0)
    st = A.acnn_conv2d_fused(d, xd, wd, bd, None, None, A.RES_NONE, A.ACT_RELU, y, ws,
                             ws.numel())
    assert st == 0
    torch.cuda.synchronize()
    assert A.acnn_last_device_status() == 0
    ref = O.conv2d(to64(x), to64(wt), to64(b), pad=1, act=O.ACT_RELU)
    assert_parity(y, ref, torch.bfloat16, "after recovery")
