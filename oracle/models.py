"""fp64 oracle forward passes of the workloads, composed from the oracle ops.

TEST INFRASTRUCTURE ONLY.  Each function restates one workload from its
description, independently of the CUDA path's layer lists; parameters are
drawn from the shared seeded generator (activation_cnn_gb300.inputs) by layer
name, so both sides use the same values.  Every stored activation is rounded
to the storage type (round to nearest even) between ops, as the GPU stores it
("storage emulation"); the arithmetic between stores is fp64.

Layer naming (shared with the generator only): stem.{0,1,2};
s{stage}.b{block}.conv{1,2,3} and .short; neck.lat{3,4,5}, neck.fpn{4,3},
neck.down{3,4}, neck.pan{4,5}; conv0a, conv0b, convblock.{i}, lastconv;
film, refine.c{0,1,2,3}.
"""
from __future__ import annotations

import numpy as np
import torch

from activation_cnn_gb300 import inputs as G

from . import oracle as O


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


class Params:
    """Draws (and caches) a layer's weight, bias and PReLU alpha by name."""

    def __init__(self, seed, layout, dtype):
        self.seed, self.layout, self.dtype = seed, layout, dtype

    def conv(self, name, c_out, c_in, k, prelu=False):
        w = _f64(G.conv_weight(self.seed, name, c_out, c_in, k, k, self.layout, self.dtype))
        b = _f64(G.conv_bias(self.seed, name, c_out))
        a = _f64(G.prelu_alpha(self.seed, name, c_out)) if prelu else None
        return w, b, a


class Runner:
    """Applies oracle ops with storage rounding after each stored result."""

    def __init__(self, params: Params, store_dtype):
        self.p, self.dt = params, store_dtype
        self.layout = params.layout

    def store(self, v):
        return O.round_storage(v, self.dt)

    def conv(self, x, name, c_out, k, s, p, act, residual=None, res_mode=O.RES_NONE):
        c_in = x.shape[3] if self.layout == O.NHWC else x.shape[1]
        w, b, a = self.p.conv(name, c_out, c_in, k, prelu=act == O.ACT_PRELU)
        return self.store(O.conv2d(x, w, b, stride=s, pad=p, act=act, alpha=a,
                                   residual=residual, res_mode=res_mode, layout=self.layout))

    def maxpool(self, x):
        return O.pool2d(x, O.MAX, 3, 2, 1, layout=self.layout)

    def avgpool(self, x):
        return self.store(O.pool2d(x, O.AVG, 2, 2, 0, layout=self.layout))

    def up2(self, x):
        h, w = (x.shape[1], x.shape[2]) if self.layout == O.NHWC else (x.shape[2], x.shape[3])
        return O.resize2d(x, O.NEAREST, 2 * h, 2 * w, layout=self.layout)

    def cat(self, a, b):
        return O.concat(a, b, layout=self.layout)


# ------------------------------------------------------------------ conv1, stem
def conv1(x):
    """conv3x3/s1/p1 16->32 + bias + ReLU, NHWC fp32."""
    r = Runner(Params(1234, O.NHWC, G.F32), O.F32)
    return r.conv(x, "conv", 32, 3, 1, 1, O.ACT_RELU)


def stem(r: Runner, x):
    """conv3x3/s2 3->32, conv3x3 32->32, conv3x3 32->64 (ReLU each), maxpool 3/2/1."""
    t = r.conv(x, "stem.0", 32, 3, 2, 1, O.ACT_RELU)
    t = r.conv(t, "stem.1", 32, 3, 1, 1, O.ACT_RELU)
    t = r.conv(t, "stem.2", 64, 3, 1, 1, O.ACT_RELU)
    return r.maxpool(t)


def stem_f32(x):
    return stem(Runner(Params(1235, O.NHWC, G.F32), O.F32), x)


# ------------------------------------------------------------------ bottleneck
def bottleneck(r: Runner, x, name, width, stride, shortcut):
    """ResNet-D bottleneck: 1x1 (ReLU) -> 3x3 with the stride (ReLU) -> 1x1; the
    shortcut (identity, 1x1 conv, or avgpool 2x2/s2 then 1x1) is added and the
    sum goes through ReLU."""
    mid = width // 4
    if shortcut == "identity":
        res = x
    elif shortcut == "conv":
        res = r.conv(x, f"{name}.short", width, 1, 1, 0, O.ACT_NONE)
    else:
        res = r.conv(r.avgpool(x), f"{name}.short", width, 1, 1, 0, O.ACT_NONE)
    t = r.conv(x, f"{name}.conv1", mid, 1, 1, 0, O.ACT_RELU)
    t = r.conv(t, f"{name}.conv2", mid, 3, stride, 1, O.ACT_RELU)
    return r.conv(t, f"{name}.conv3", width, 1, 1, 0, O.ACT_RELU, residual=res,
                  res_mode=O.RES_ADD_THEN_ACT)


def block(x, variant):
    r = Runner(Params(1236, O.NHWC, G.BF16), O.BF16)
    if variant == "identity":
        return bottleneck(r, x, "id", 256, 1, "identity")
    return bottleneck(r, x, "down", 512, 2, "pool")


# ------------------------------------------------------------------ backbone + neck
def csp(r: Runner, x, name, blocks=3, hidden=256):
    """P1 RtDetrGpu::csp: a = conv1(x) (1x1 + SiLU); per RepVGG bottleneck
    a = SiLU(conv3x3(a) + conv1x1(a)) (branches without activation); out =
    a + conv2(x) (conv2 1x1 + SiLU, plain add).  Each conv's output is stored
    (bf16) before the next op reads it."""
    S = O.ACT_SILU
    a = r.conv(x, f"{name}.conv1", hidden, 1, 1, 0, S)
    for i in range(blocks):
        q = r.conv(a, f"{name}.rep{i}.conv1x1", hidden, 1, 1, 0, O.ACT_NONE)
        a = r.conv(a, f"{name}.rep{i}.conv3x3", hidden, 3, 1, 1, S, residual=q,
                   res_mode=O.RES_ADD_THEN_ACT)
    return r.conv(x, name, 256, 1, 1, 0, S, residual=a, res_mode=O.RES_ACT_THEN_ADD)


def backbone(x, neck="fusion"):
    """ResNet-D-50 (3/4/6/3 blocks, widths 256/512/1024/2048; stage 1 shortcut a
    1x1 conv, later stages avgpool + 1x1; stride on the first 3x3 of stages 2-4)
    and the neck: SiLU lateral 1x1s to 256; top-down nearest-2x + concat
    [upsampled, lateral] + SiLU conv3x3 to 256; bottom-up SiLU conv3x3/s2 +
    concat [downsampled, top-down map] + SiLU conv3x3.  Returns (F3, N4, N5)."""
    r = Runner(Params(1238, O.NHWC, G.BF16), O.BF16)
    t = stem(r, x)
    feats = []
    for si, (blocks, width, stride, first) in enumerate(
            [(3, 256, 1, "conv"), (4, 512, 2, "pool"), (6, 1024, 2, "pool"), (3, 2048, 2, "pool")]):
        for bi in range(blocks):
            t = bottleneck(r, t, f"s{si + 1}.b{bi}", width, stride if bi == 0 else 1,
                           first if bi == 0 else "identity")
        feats.append(t)
    c3, c4, c5 = feats[1], feats[2], feats[3]
    S = O.ACT_SILU
    lat3 = r.conv(c3, "neck.lat3", 256, 1, 1, 0, S)
    lat4 = r.conv(c4, "neck.lat4", 256, 1, 1, 0, S)
    f5 = r.conv(c5, "neck.lat5", 256, 1, 1, 0, S)

    def fuse(x, name):
        if neck == "csp":
            return csp(r, x, name)
        return r.conv(x, name, 256, 3, 1, 1, S)

    f4 = fuse(r.cat(r.up2(f5), lat4), "neck.fpn4")
    f3 = fuse(r.cat(r.up2(f4), lat3), "neck.fpn3")
    d3 = r.conv(f3, "neck.down3", 256, 3, 2, 1, S)
    n4 = fuse(r.cat(d3, f4), "neck.pan4")
    d4 = r.conv(n4, "neck.down4", 256, 3, 2, 1, S)
    n5 = fuse(r.cat(d4, f5), "neck.pan5")
    return f3, n4, n5


# ------------------------------------------------------------------ frame stack
def frame(rgba0, rgba1, t=0.5, c1=120, c2=240, flow_out=False):
    """rt.js run() up to the x8 upsample: prep -> prelu(conv s2) x2 -> 8 x conv +
    PReLU with the map entering the 8 added after the 8th PReLU -> deconv 4x4/s2
    -> bilinear x8.  NCHW fp16 storage.  With flow_out the last step is the
    flow-out stage instead, returning the interpolated [H, W, 4] RGBA8 frame."""
    r = Runner(Params(1237, O.NCHW, G.F16), O.F16)
    xq = r.store(O.prep_quarter(rgba0, rgba1, t))[None]
    P = O.ACT_PRELU
    a = r.conv(xq, "conv0a", c1, 3, 2, 1, P)
    f = r.conv(a, "conv0b", c2, 3, 2, 1, P)
    skip = f
    for i in range(8):
        if i < 7:
            f = r.conv(f, f"convblock.{i}", c2, 3, 1, 1, P)
        else:
            f = r.conv(f, f"convblock.{i}", c2, 3, 1, 1, P, residual=skip,
                       res_mode=O.RES_ACT_THEN_ADD)
    w = _f64(G.deconv_weight(1237, "lastconv", c2, 5, 4))
    b = _f64(G.conv_bias(1237, "lastconv", 5))
    tmp8 = r.store(O.deconv2d(f, w, b))
    h, wd = rgba0.shape[0], rgba0.shape[1]
    if flow_out:
        # rt.js wgslFlowOut on the fp16-stored map, in binary32 as on the page
        return O.flow_out(tmp8[0].astype(np.float32), rgba0, rgba1)
    return r.store(O.resize2d(tmp8, O.BILINEAR, h, wd, layout=O.NCHW))


def frame_tfact(rgba0, rgba1, ts=(0.25, 0.5, 0.75), c1=120, c2=240, hn=64, rc=32):
    """rt.js tfact2, prepPair then runT per t: the t-free trunk (six prep planes
    -> prelu(conv s2) x2 -> convblocks 0..5) once, then per t: FiLM(t) ->
    convblocks 6, 7 (7 adding the map that entered convblock 0 after its
    PReLU) -> deconv 4x4/s2 -> refine prep -> three conv3x3 + PReLU (zero pad)
    -> refine out (replicate pad, 2 sigmoid - 1) -> flow-out with that residual.
    NCHW fp16 storage; the refine residual is fp32 (its buffer type on the
    page); the flow-out stage runs in binary32.  One RGBA8 frame per t."""
    seed = 1238
    r = Runner(Params(seed, O.NCHW, G.F16), O.F16)
    xq = r.store(O.prep_quarter(rgba0, rgba1, 0.0)[:6])[None]
    P = O.ACT_PRELU
    a = r.conv(xq, "conv0a", c1, 3, 2, 1, P)
    feat0 = r.conv(a, "conv0b", c2, 3, 2, 1, P)
    trunk = feat0
    for i in range(6):
        trunk = r.conv(trunk, f"convblock.{i}", c2, 3, 1, 1, P)
    w0, b0, w2, b2 = (_f64(t) for t in G.film_mlp(seed, "film", c2, hn))
    wdc = _f64(G.deconv_weight(seed, "lastconv", c2, 5, 4))
    bdc = _f64(G.conv_bias(seed, "lastconv", 5))
    wro = _f64(G.refine_out_weight(seed, "refine.c3", rc))
    bro = _f64(G.conv_bias(seed, "refine.c3", 3))
    outs = []
    for t in ts:
        f = r.store(O.film(trunk[0], t, w0, b0, w2, b2))[None]
        f = r.conv(f, "convblock.6", c2, 3, 1, 1, P)
        f = r.conv(f, "convblock.7", c2, 3, 1, 1, P, residual=feat0, res_mode=O.RES_ACT_THEN_ADD)
        tmp8 = r.store(O.deconv2d(f, wdc, bdc))
        rin = r.store(O.refine_prep(tmp8[0], rgba0, rgba1))[None]
        x = r.conv(rin, "refine.c0", rc, 3, 1, 1, P)
        x = r.conv(x, "refine.c1", rc, 3, 1, 1, P)
        x = r.conv(x, "refine.c2", rc, 3, 1, 1, P)
        res = O.round_storage(O.refine_out(x[0], wro, bro), O.F32).astype(np.float32)
        outs.append(O.flow_out(tmp8[0].astype(np.float32), rgba0, rgba1, res=res))
    return outs
