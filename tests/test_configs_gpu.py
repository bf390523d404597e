"""The workloads end to end, CUDA graphs vs the fp64 oracle.

* conv1, stem, block (both variants): full size, end to end against the
  oracle forward pass with storage emulation (every stored map rounded).
* backbone (both necks) and the frame stacks: end to end at full size (the
  launch configuration bench.py times) against the oracle's forward pass with
  storage emulation, and layer by layer, teacher-forced (each conv's oracle is
  fed the GPU's stored input): every output pixel of every conv of the
  backbone and frame stacks, sampled pixels for the CSP-neck variant's 92
  convs; the memory-bound ops on whole maps.  Also end to end at a reduced
  size the oracle finishes in a second or two.
"""
import numpy as np
import pytest
import torch

from activation_cnn_gb300 import acnn as A
from activation_cnn_gb300 import inputs as G
from activation_cnn_gb300 import network as N
from oracle import models as M
from oracle import oracle as O
from tests.parity import assert_bitexact, assert_bytes_boundary, assert_parity, metrics, to64

pytestmark = pytest.mark.gpu


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


def run_graph(net):
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        net.run_eager(s)
    s.synchronize()
    net.capture(s)
    for t in net.output_tensors():
        t.zero_()
    torch.cuda.synchronize()
    net.replay(s)
    s.synchronize()
    outs = [t.clone() for t in net.output_tensors()]
    net.release()
    return outs


def assert_maps(outs, refs, dtype):
    for i, (g, r) in enumerate(zip(outs, refs)):
        m = metrics(g, r.reshape(g.shape))
        print(f"map {i}: {m}")
        if dtype == torch.float32:
            assert m["rel_l2"] <= 1e-5 and m["max_abs"] <= 1e-4, (i, m)
        else:
            assert m["rel_l2"] <= 2e-2 and m["cos"] >= 0.9999, (i, m)


def test_conv1_full():
    net = N.conv1_net()
    (y,) = run_graph(net)
    ref = M.conv1(to64(net.inputs["x"]))
    assert_maps([y], [ref], torch.float32)


def test_stem_full():
    net = N.stem_net()
    (y,) = run_graph(net)
    assert tuple(y.shape) == (1, 160, 160, 64)
    ref = M.stem_f32(to64(net.inputs["x"]))
    assert_maps([y], [ref], torch.float32)


@pytest.mark.parametrize("variant", ["identity", "downsample"])
def test_block_full(variant):
    net = N.block_net(variant=variant)
    (y,) = run_graph(net)
    ref = M.block(to64(net.inputs["x"]), variant)
    assert_maps([y], [ref], torch.bfloat16)


def test_frame_reduced_end_to_end():
    net = N.frame_net(h=128, w=192)
    (y,) = run_graph(net)
    ref = M.frame(net.inputs["frame0"].cpu().numpy(), net.inputs["frame1"].cpu().numpy())
    assert_maps([y], [ref], torch.float16)


def test_frame_out_reduced_end_to_end():
    """The frame stack ending in the flow-out stage, against the oracle's stack
    (fp64 convs with fp16 storage, binary32 flow-out).  The two 1/8-resolution
    maps differ by fp16 storage-rounding noise, and warping random-noise frames
    turns a flow difference of d pixels into byte differences of up to ~255*d,
    so the bytes are compared statistically; the flow-out kernel itself is
    checked byte for byte in test_ops_gpu.py."""
    net = N.frame_net(h=128, w=192, flow_out=True)
    (y,) = run_graph(net)
    f0, f1 = net.inputs["frame0"].cpu().numpy(), net.inputs["frame1"].cpu().numpy()
    ref = M.frame(f0, f1, flow_out=True)
    got = y.cpu().numpy()
    assert got.shape == ref.shape == (128, 192, 4)
    assert (got[..., 3] == 255).all()
    d = np.abs(got[..., :3].astype(np.int32) - ref[..., :3].astype(np.int32))
    print(f"frame_out: exact {np.mean(d == 0):.4f}, within 1 {np.mean(d <= 1):.4f}, "
          f"mean {d.mean():.4f}, max {d.max()}")
    # bound: the maps agree to fp16 storage rounding (about 1e-3 relative), the
    # flows are scaled by 8, and a flow difference of d pixels moves a byte of a
    # random-noise frame by up to 255 * d -- so a few bytes per thousand may move
    # by 2 and none by more than 4; most agree exactly
    assert d.max() <= 4 and np.mean(d <= 1) >= 0.995 and d.mean() <= 0.3 and \
        np.mean(d == 0) >= 0.75, (np.mean(d == 0), np.mean(d <= 1), d.mean(), d.max())


def _tfact_stages(net, ts, h, w):
    """Teacher-forced check of the t-factored stack's non-conv stages on the
    GPU's own stored inputs: FiLM and the refine pair against the fp64 oracle,
    the flow-out bytes (with the refine residual) under the byte-boundary rule."""
    T = net.tensors
    f0, f1 = net.inputs["frame0"].cpu().numpy(), net.inputs["frame1"].cpu().numpy()
    prm = [to64(p) for p in net.params["film"]]
    w3, b3, _ = net.params["refine.c3"]
    for i, t in enumerate(ts):
        sfx = f"@t{i}"
        assert_parity(T["film" + sfx][0], O.film(to64(T["convblock.5"][0]), t, *prm),
                      torch.float16, "film" + sfx)
        tmp8 = to64(T["tmp8" + sfx][0])
        assert_parity(T["rin" + sfx][0], O.refine_prep(tmp8, f0, f1), torch.float16,
                      "refine_prep" + sfx)
        assert_parity(T["rres" + sfx][0], O.refine_out(to64(T["refine.c2" + sfx][0]), to64(w3),
                                                       to64(b3)), torch.float32,
                      "refine_out" + sfx)
        ref, pre = O.flow_out(tmp8.astype(np.float32), f0, f1,
                              res=T["rres" + sfx][0].cpu().numpy(), with_pre=True)
        assert_bytes_boundary(T["out" + sfx], ref, pre, "flow_out" + sfx)


def test_frame_tfact_reduced_end_to_end():
    """The t-factored stack with the refine head at 128x192, three timesteps.

    Teacher-forced, every stage matches (convs on all pixels, FiLM and the
    refine pair to parity, flow-out bytes under the byte-boundary rule).  End to end against the
    oracle's stack the bytes are compared statistically, as for frame_out, with
    one more noise source: the fp32 residual comes out of three fp16-stored
    convs (relative noise ~2^-11 per store, variance-preserving weights) and
    2 sigmoid - 1 (slope <= 1/2), so it differs by a few 1e-3, which moves a
    byte by at most about 1 on top of the warp's moves."""
    ts = (0.25, 0.5, 0.75)
    net = N.frame_tfact_net(h=128, w=192, ts=ts)
    outs = run_graph(net)
    assert len(outs) == 3 and all(tuple(o.shape) == (128, 192, 4) for o in outs)
    assert check_layers(net, samples=10**6) == 8 + 3 * 5
    _tfact_stages(net, ts, 128, 192)
    f0, f1 = net.inputs["frame0"].cpu().numpy(), net.inputs["frame1"].cpu().numpy()
    refs = M.frame_tfact(f0, f1, ts)
    for i, (y, ref) in enumerate(zip(outs, refs)):
        got = y.cpu().numpy()
        assert (got[..., 3] == 255).all()
        d = np.abs(got[..., :3].astype(np.int32) - ref[..., :3].astype(np.int32))
        print(f"frame_tfact t={ts[i]}: exact {np.mean(d == 0):.4f}, within 1 "
              f"{np.mean(d <= 1):.4f}, mean {d.mean():.4f}, max {d.max()}")
        assert d.max() <= 6 and np.mean(d <= 1) >= 0.98 and d.mean() <= 0.6, \
            (ts[i], np.mean(d == 0), np.mean(d <= 1), d.mean(), d.max())
    # different timesteps give different frames
    assert not torch.equal(outs[0], outs[2])


def test_backbone_reduced_end_to_end():
    net = N.backbone_net(n=1, h=128, w=160)
    outs = run_graph(net)
    refs = M.backbone(to64(net.inputs["x"]))
    assert [tuple(o.shape) for o in outs] == [(1, 16, 20, 256), (1, 8, 10, 256), (1, 4, 5, 256)]
    assert_maps(outs, refs, torch.bfloat16)


def test_backbone_csp_reduced_end_to_end():
    """The neck with P1's CSP/RepVGG blocks in place of the single fusion convs."""
    net = N.backbone_net(n=1, h=128, w=160, neck="csp")
    outs = run_graph(net)
    refs = M.backbone(to64(net.inputs["x"]), neck="csp")
    assert [tuple(o.shape) for o in outs] == [(1, 16, 20, 256), (1, 8, 10, 256), (1, 4, 5, 256)]
    assert_maps(outs, refs, torch.bfloat16)


# ------------------------------------------------------------------ full size, per layer
def _sample_pixels(n, oh, ow, k, rng):
    if k >= n * oh * ow:  # every pixel
        return [(b, y, x) for b in range(n) for y in range(oh) for x in range(ow)]
    pts = {(0, 0, 0), (n - 1, oh - 1, ow - 1), (0, oh - 1, 0), (n - 1, 0, ow - 1)}
    while len(pts) < k:
        pts.add((int(rng.integers(n)), int(rng.integers(oh)), int(rng.integers(ow))))
    return sorted(pts)


def check_layers(net, samples=48):
    """Each conv of a graph-replayed net against the oracle fed the GPU's stored
    input (teacher-forced): on `samples` pixels (all channels), or on every
    output pixel with samples=None."""
    rng = np.random.default_rng(0)
    T = net.tensors
    tdt = {G.F32: torch.float32, G.F16: torch.float16, G.BF16: torch.bfloat16}[net.dtype]
    checked = 0
    for op in net.ops:
        if op.kind != "conv":
            continue
        s = op.spec
        x_name = _input_of(net, op)
        if isinstance(x_name, tuple):  # a concat folded into the conv
            x = O.concat(to64(T[x_name[0]]), to64(T[x_name[1]]), layout=net.layout)
        else:
            x = to64(T[x_name])
        y = T[s.name]
        w, b, al = net.params[s.name]
        res = None
        if s.res_mode != A.RES_NONE:
            res = to64(T[_residual_of(net, op)])
        kw = dict(stride=s.stride, pad=s.pad, act=s.act, alpha=None if al is None else to64(al),
                  residual=res, res_mode=s.res_mode, layout=net.layout)
        if samples is None:
            ref = O.conv2d(x, to64(w), to64(b), **kw)
            assert_parity(y, ref, tdt, s.name)
        else:
            pts = _sample_pixels(net.batch, s.oh, s.ow, samples, rng)
            ref = O.conv2d_points(x, to64(w), to64(b), pts, **kw)
            yg = to64(y)
            if net.layout == G.NHWC:
                got = np.stack([yg[n, oy, ox, :] for n, oy, ox in pts])
            else:
                got = np.stack([yg[n, :, oy, ox] for n, oy, ox in pts])
            assert_parity(got, ref, tdt, s.name)
        checked += 1
    return checked


def _input_of(net, op):
    return net.conv_inputs[op.spec.name]


def _residual_of(net, op):
    return net.conv_residuals[op.spec.name]


def test_backbone_full_size():
    """The 8x640x640 workload: end to end against the oracle's forward pass with
    bf16 storage emulation; then every one of the 64 convs teacher-forced on
    every output pixel (so every plan the backbone uses -- each tile width,
    256-row tiles, split-K, resident weights, the folded concats -- is checked
    on all its tiles), and the memory-bound ops on whole maps."""
    net = N.backbone_net()
    outs = run_graph(net)
    assert [tuple(o.shape) for o in outs] == [(8, 80, 80, 256), (8, 40, 40, 256), (8, 20, 20, 256)]
    refs = M.backbone(to64(net.inputs["x"]))
    assert_maps(outs, refs, torch.bfloat16)
    # the graph replay left every intermediate map in place: check each layer on it
    assert check_layers(net, samples=None) == 64
    T = net.tensors
    assert_bitexact(T["stem.pool"], O.pool2d(to64(T["stem.2"]), O.MAX, 3, 2, 1), "maxpool")
    assert_bitexact(T["neck.up5"], O.resize2d(to64(T["neck.lat5"]), O.NEAREST, 40, 40), "up5")
    assert_bitexact(T["neck.up4"], O.resize2d(to64(T["neck.fpn4"]), O.NEAREST, 80, 80), "up4")
    # the stage-to-stage average pools, written by the conv that produces their
    # input (acnn_conv2d_fused_pool2): bit for bit the pool kernel's result on
    # that conv's stored output, and within tolerance of the oracle
    assert sorted(net.pooled.values()) == ["s1.b2.conv3", "s2.b3.conv3", "s3.b5.conv3"]
    for pooled, src in net.pooled.items():
        assert_bitexact(T[pooled], A.pool2d(T[src], A.POOL_AVG, 2, 2, 0), pooled)
        assert_parity(T[pooled], O.pool2d(to64(T[src]), O.AVG, 2, 2, 0), torch.bfloat16, pooled)


def test_backbone_full_size_replays_are_bitwise_identical():
    """Two replays of the 8x640x640 graphs give the same bits in every map the
    step writes: no kernel depends on timing or arrival order (split-K sums its
    partial tiles in split order, every other output has one writer)."""
    net = N.backbone_net()
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        net.run_eager(s)
    s.synchronize()
    net.capture(s)
    names = [n for n, t in net.tensors.items() if t is not None and not n.endswith(".ws")
             and n not in net.inputs]
    snaps = []
    for _ in range(2):
        for n in names:
            net.tensors[n].fill_(float("nan")) if net.tensors[n].is_floating_point() else None
        torch.cuda.synchronize()
        net.replay(s)
        s.synchronize()
        snaps.append({n: net.tensors[n].clone() for n in names})
    net.release()
    for n in names:
        assert torch.equal(snaps[0][n], snaps[1][n]), n
    assert A.acnn_last_device_status() == 0


def test_backbone_csp_full_size():
    """The CSP-neck variant at 8x640x640: end to end against the oracle, and its
    92 convs teacher-forced on sampled pixels."""
    net = N.backbone_net(neck="csp")
    outs = run_graph(net)
    refs = M.backbone(to64(net.inputs["x"]), neck="csp")
    assert_maps(outs, refs, torch.bfloat16)
    assert check_layers(net, samples=24) == 92


def test_frame_full_size():
    """1088x1920: end to end against the oracle's stack (fp16 storage
    emulation), then every conv teacher-forced on every output pixel and the
    other stages on whole maps."""
    net = N.frame_net()
    (flow,) = run_graph(net)
    assert tuple(flow.shape) == (1, 5, 1088, 1920)
    f0, f1 = net.inputs["frame0"].cpu().numpy(), net.inputs["frame1"].cpu().numpy()
    assert_maps([flow], [M.frame(f0, f1)], torch.float16)
    assert check_layers(net, samples=None) == 10
    T = net.tensors
    assert_parity(T["xq"], O.prep_quarter(f0, f1, 0.5)[None], torch.float16, "prep")
    w, b, _ = net.params["lastconv"]
    ref = O.deconv2d(to64(T["convblock.7"]), to64(w), to64(b))
    assert_parity(T["tmp8"], ref, torch.float16, "deconv")
    ref = O.resize2d(to64(T["tmp8"]), O.BILINEAR, 1088, 1920, layout=O.NCHW)
    assert_parity(flow, ref, torch.float16, "bilinear x8")


def _byte_stats(got, ref):
    d = np.abs(got[..., :3].astype(np.int32) - ref[..., :3].astype(np.int32))
    return d, np.mean(d == 0), np.mean(d <= 1), d.mean(), d.max()


def test_frame_out_full_size():
    """The frame stack ending in the flow-out stage at 1088x1920, end to end
    against the oracle's stack (bytes compared statistically, as at the
    reduced size: the 1/8-resolution maps differ by fp16 storage noise, which
    the warp of random-noise frames turns into byte differences), and the
    flow-out stage teacher-forced on the GPU's own map under the byte-boundary
    rule."""
    net = N.frame_net(flow_out=True)
    (y,) = run_graph(net)
    f0, f1 = net.inputs["frame0"].cpu().numpy(), net.inputs["frame1"].cpu().numpy()
    ref = M.frame(f0, f1, flow_out=True)
    got = y.cpu().numpy()
    assert got.shape == ref.shape == (1088, 1920, 4)
    assert (got[..., 3] == 255).all()
    d, eq, le1, mean, mx = _byte_stats(got, ref)
    print(f"frame_out full: exact {eq:.4f}, within 1 {le1:.4f}, mean {mean:.4f}, max {mx}")
    assert mx <= 4 and le1 >= 0.995 and mean <= 0.3 and eq >= 0.75, (eq, le1, mean, mx)
    tmp8 = net.tensors["tmp8"][0].float().cpu().numpy()
    r, pre = O.flow_out(tmp8, f0, f1, with_pre=True)
    assert_bytes_boundary(y, r, pre, "flow_out (teacher-forced)")


def test_frame_tfact_full_size():
    """1088x1920, three timesteps: end to end against the oracle's stack (bytes
    statistically, as at the reduced size), then teacher-forced the 23 convs on
    every output pixel and the other stages on whole maps."""
    ts = (0.25, 0.5, 0.75)
    net = N.frame_tfact_net(ts=ts)
    outs = run_graph(net)
    assert [tuple(o.shape) for o in outs] == [(1088, 1920, 4)] * 3
    f0, f1 = net.inputs["frame0"].cpu().numpy(), net.inputs["frame1"].cpu().numpy()
    refs = M.frame_tfact(f0, f1, ts=ts)
    for i, (y, ref) in enumerate(zip(outs, refs)):
        got = y.cpu().numpy()
        assert (got[..., 3] == 255).all()
        d, eq, le1, mean, mx = _byte_stats(got, ref)
        print(f"frame_tfact full t={ts[i]}: exact {eq:.4f}, within 1 {le1:.4f}, "
              f"mean {mean:.4f}, max {mx}")
        assert mx <= 6 and le1 >= 0.98 and mean <= 0.6, (ts[i], eq, le1, mean, mx)
    assert check_layers(net, samples=None) == 8 + 3 * 5
    _tfact_stages(net, ts, 1088, 1920)
