"""Layer graphs of the workloads, run through the C ABI and replayed as CUDA graphs.

A ``Net`` is an ordered list of ops grouped into sections.  Each op is one
ABI call on buffers allocated once (PyTorch supplies the device memory); a
section is captured once into a CUDA graph with the ABI's section runner and
replayed per step -- the GPU form of rtdetr_gpu.rs's Recorder (one submit per
section) and rt.js's single command buffer per frame.

Workloads (seeded, synthetic; the parameters come from
activation_cnn_gb300.inputs by layer name):
  conv1   one conv3x3/s1/p1 16->32 + ReLU, NHWC fp32, 1x32x32
  stem    conv3x3/s2 3->32, conv3x3 32->32, conv3x3 32->64 (+ReLU each),
          maxpool 3/2/1; NHWC fp32, 1x640x640x3
  block   ResNet bottleneck at 4x80x80x256 bf16, identity variant and the
          stride-2 downsample variant with an avgpool + 1x1 shortcut
  frame   frame-interpolation stack, NCHW fp16, two 1920x1088 RGBA8 frames
  frame_out  the same stack ending in the flow-out stage (interpolated RGBA8 frame)
  backbone  ResNet-D-50 (3/4/6/3 bottlenecks) + top-down/bottom-up neck,
          NHWC bf16, 8x640x640x3
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import acnn as A
from . import inputs as G

TDT = G.TORCH_DTYPE


@dataclass
class ConvSpec:
    name: str
    c_in: int
    c_out: int
    k: int
    stride: int
    pad: int
    act: int
    h: int  # input height
    w: int  # input width
    res_mode: int = A.RES_NONE
    param: str = ""  # name the weights are drawn under (default: name)

    @property
    def oh(self):
        return (self.h + 2 * self.pad - self.k) // self.stride + 1

    @property
    def ow(self):
        return (self.w + 2 * self.pad - self.k) // self.stride + 1


@dataclass
class Op:
    kind: str                # conv | pool | resize | concat | deconv | prep
    section: str
    fn: object = None        # callable(stream) issuing the ABI call(s)
    flops: float = 0.0       # algorithmic FLOPs of one call
    bytes: float = 0.0       # algorithmic bytes (inputs read once + output written once)
    label: str = ""
    spec: object = None
    launches: int = 1        # kernels one call launches (non-conv ops)
    # Parallel branch: an op with side = k > 0 runs on the net's side stream k
    # (forked from the main stream at the first such op of a section); a `join`
    # op waits on the main stream for every side op before it.  A section ends
    # joined.
    side: int = 0
    join: bool = False


@dataclass
class Net:
    name: str
    batch: int
    dtype: int
    layout: int
    ops: list = field(default_factory=list)
    tensors: dict = field(default_factory=dict)
    inputs: dict = field(default_factory=dict)   # name -> device tensor fed per step
    outputs: list = field(default_factory=list)  # names of the output tensors
    params: dict = field(default_factory=dict)   # name -> (cpu tensors) for reference checks
    graphs: list = field(default_factory=list)   # [(section, Section)]
    order: list = field(default_factory=list)    # section names in execution order
    conv_inputs: dict = field(default_factory=dict)     # conv name -> input tensor name(s)
    conv_residuals: dict = field(default_factory=dict)  # conv name -> residual tensor name
    pooled: dict = field(default_factory=dict)  # pooled map written by a conv -> that conv's name
    upsampled: dict = field(default_factory=dict)  # 2x-upsampled map written by a conv -> its name

    # ------------------------------------------------------------ execution
    def sections(self):
        return list(self.order)

    def side_stream(self, device, k=1):
        """Side stream k (created once per net)."""
        if getattr(self, "_sides", None) is None:
            self._sides = {}
        if k not in self._sides:
            self._sides[k] = torch.cuda.Stream(device=device)
        return self._sides[k]

    def enqueue(self, stream, section=None, hook=None):
        """Enqueue the ops (of one section, or all) on `stream`, side ops on their
        side streams between a fork and a join (events: under stream capture they
        become parallel branches of the section's graph).  hook(op, stream, when)
        runs before ("pre") and after ("post") each op on the stream it uses."""
        pending = {}  # side id -> its stream, forked and not yet joined

        def join_all():
            for side in pending.values():
                ev = torch.cuda.Event()
                ev.record(side)
                stream.wait_event(ev)
            pending.clear()

        for op in self.ops:
            if section is not None and op.section != section:
                continue
            if op.join:
                join_all()
            target = stream
            if op.side:
                if op.side not in pending:
                    side = self.side_stream(stream.device, op.side)
                    ev = torch.cuda.Event()
                    ev.record(stream)
                    side.wait_event(ev)
                    pending[op.side] = side
                target = pending[op.side]
            if hook:
                hook(op, target, "pre")
            op.fn(target)
            if hook:
                hook(op, target, "post")
        join_all()

    def run_eager(self, stream=None, section=None):
        s = stream if stream is not None else torch.cuda.current_stream()
        self.enqueue(s, section)

    def capture(self, stream):
        """Record one CUDA graph per section on `stream` (ops must have run once)."""
        self.release()
        for sec in self.order:
            g = A.Section(stream)
            with torch.cuda.stream(stream):
                with g:
                    self.run_eager(stream, sec)
            self.graphs.append((sec, g))

    def replay(self, stream):
        for _, g in self.graphs:
            g.launch(stream)

    def release(self):
        for _, g in self.graphs:
            g.close()
        self.graphs = []

    # ------------------------------------------------------------ accounting
    def conv_flops(self):
        return sum(op.flops for op in self.ops if op.kind == "conv")

    def total_flops(self):
        return sum(op.flops for op in self.ops)

    def output_tensors(self):
        return [self.tensors[n] for n in self.outputs]


def _conv_flops(n, s: ConvSpec):
    return 2.0 * n * s.oh * s.ow * s.c_out * s.c_in * s.k * s.k


class Builder:
    """Allocates buffers, draws parameters and appends ABI ops to a Net."""

    def __init__(self, net: Net, seed: int, device="cuda"):
        self.net = net
        self.seed = seed
        self.device = device
        self.section = "main"
        self.es = 4 if net.dtype == G.F32 else 2

    def side(self, k=1):
        """Ops appended inside `with b.side(k):` run on the net's side stream k."""
        b = self

        class _Side:
            def __enter__(self_):
                self_.start = len(b.net.ops)

            def __exit__(self_, *exc):
                for op in b.net.ops[self_.start:]:
                    op.side = k
                return False
        return _Side()

    def set_section(self, name):
        self.section = name
        if name not in self.net.order:
            self.net.order.append(name)

    def buffer(self, name, c, h, w, dtype=None, n=None):
        n = self.net.batch if n is None else n
        dt = TDT[self.net.dtype if dtype is None else dtype]
        shape = G.activation_shape(self.net.layout, n, c, h, w)
        t = torch.empty(shape, dtype=dt, device=self.device)
        self.net.tensors[name] = t
        return t

    def conv(self, src, spec: ConvSpec, residual=None, out=None, pool2=None, up2=None,
             nhwc_copy=False):
        """nhwc_copy (NCHW convs on the tensor cores): also write an NHWC copy of
        the output (tensor f"{name}.nhwc"); a conv whose input has such a copy
        reads it instead of staging the input itself."""
        net = self.net
        if pool2:
            return self._conv_pool2(src, spec, residual, pool2)
        if up2:
            return self._conv_up2(src, None, spec, residual, up2)
        x = net.tensors[src]
        pn = spec.param or spec.name
        w = G.conv_weight(self.seed, pn, spec.c_out, spec.c_in, spec.k, spec.k, net.layout,
                          net.dtype)
        b = G.conv_bias(self.seed, pn, spec.c_out)
        al = G.prelu_alpha(self.seed, pn, spec.c_out) if spec.act == A.ACT_PRELU else None
        net.params[spec.name] = (w, b, al)
        wd, bd = w.to(self.device), b.to(self.device)
        ald = al.to(self.device) if al is not None else None
        y = self.buffer(out or spec.name, spec.c_out, spec.oh, spec.ow)
        res = net.tensors[residual] if residual else None
        d = A.conv_desc(x, spec.c_out, spec.k, spec.k, spec.stride, spec.pad, net.layout)
        path = A.acnn_conv2d_path(d)
        # convs whose weights would be restaged on every call (the packed path,
        # NCHW convs on the tensor cores) take them prepacked once, here
        staged = path == 3 or (path in (1, 2) and net.layout == G.NCHW)
        if staged:
            wd = A.conv2d_prepack(d, wd)
            torch.cuda.synchronize()
            ws_bytes = A.acnn_conv2d_prepacked_workspace_size(d)
        else:
            ws_bytes = A.acnn_conv2d_workspace_size(d)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=self.device) if ws_bytes else None
        net.tensors[spec.name + ".ws"] = ws
        res_mode = spec.res_mode if residual else A.RES_NONE
        net.conv_inputs[spec.name] = src
        if residual:
            net.conv_residuals[spec.name] = residual
        # NHWC copies along a chain of NCHW tensor-core convs: the input's copy
        # (written by the conv that produced it) spares this conv its staging
        # transpose; this conv writes its own output's copy when asked to
        tc_nchw = net.layout == G.NCHW and path in (1, 2)
        x_copy = net.tensors.get(src + ".nhwc") if tc_nchw else None
        y_copy = None
        if nhwc_copy and net.layout == G.NCHW and path in (1, 2, 3):
            y_copy = torch.empty((net.batch, spec.oh, spec.ow, spec.c_out), dtype=y.dtype,
                                 device=self.device)
            net.tensors[(out or spec.name) + ".nhwc"] = y_copy
        if x_copy is not None or y_copy is not None:
            def fn(stream, d=d, x=x, wd=wd, bd=bd, ald=ald, res=res, y=y, ws=ws, res_mode=res_mode,
                   x_copy=x_copy, y_copy=y_copy):
                A.check(A.acnn_conv2d_fused_prepacked_staged(d, x, x_copy, wd, bd, ald, res,
                                                             res_mode, spec.act, y, y_copy, ws,
                                                             ws_bytes, stream), spec.name)
        else:
            call = A.acnn_conv2d_fused_prepacked if staged else A.acnn_conv2d_fused

            def fn(stream, d=d, x=x, wd=wd, bd=bd, ald=ald, res=res, y=y, ws=ws, res_mode=res_mode):
                A.check(call(d, x, wd, bd, ald, res, res_mode, spec.act, y, ws, ws_bytes, stream),
                        spec.name)

        n = net.batch
        byts = (x.numel() + w.numel() + y.numel() + (y.numel() if res is not None else 0)) * \
            self.es + 4 * spec.c_out
        # kernels per call: the conv, plus the activation staging (NCHW -> NHWC
        # copy or im2col pack) of a staged conv unless its input's copy exists
        if y_copy is not None:
            byts += y.numel() * self.es
        net.ops.append(Op("conv", self.section, fn, _conv_flops(n, spec), byts, spec.name, spec,
                          launches=2 if staged and x_copy is None else 1))
        return out or spec.name

    def _conv_pool2(self, src, spec: ConvSpec, residual, pool_name):
        """A 1x1 NHWC conv that also writes the 2x2/s2 average pool of its output
        (tensor pool_name), for the next stage's shortcut (acnn_conv2d_fused_pool2)."""
        net = self.net
        x = net.tensors[src]
        w = G.conv_weight(self.seed, spec.param or spec.name, spec.c_out, spec.c_in, 1, 1,
                          net.layout, net.dtype)
        b = G.conv_bias(self.seed, spec.param or spec.name, spec.c_out)
        al = G.prelu_alpha(self.seed, spec.param or spec.name, spec.c_out) \
            if spec.act == A.ACT_PRELU else None
        net.params[spec.name] = (w, b, al)
        wd, bd = w.to(self.device), b.to(self.device)
        ald = al.to(self.device) if al is not None else None
        y = self.buffer(spec.name, spec.c_out, spec.oh, spec.ow)
        yp = self.buffer(pool_name, spec.c_out, spec.oh // 2, spec.ow // 2)
        res = net.tensors[residual] if residual else None
        res_mode = spec.res_mode if residual else A.RES_NONE
        d = A.conv_desc(x, spec.c_out, 1, 1, 1, 0, net.layout)
        net.conv_inputs[spec.name] = src
        if residual:
            net.conv_residuals[spec.name] = residual
        net.pooled[pool_name] = spec.name

        def fn(stream):
            A.check(A.acnn_conv2d_fused_pool2(d, x, wd, bd, ald, res, res_mode, spec.act, y, yp,
                                              stream), spec.name)

        byts = (x.numel() + w.numel() + y.numel() + yp.numel() +
                (y.numel() if res is not None else 0)) * self.es + 4 * spec.c_out
        net.ops.append(Op("conv", self.section, fn, _conv_flops(net.batch, spec), byts, spec.name,
                          spec))
        return spec.name

    def _conv_up2(self, src_a, src_b, spec: ConvSpec, residual, up_name):
        """An NHWC conv (over [src_a | src_b] when src_b is given) that also
        writes the nearest 2x upsample of its output (tensor up_name)
        (acnn_conv2d_fused_up2)."""
        net = self.net
        xa = net.tensors[src_a]
        xb = net.tensors[src_b] if src_b else None
        ca = xa.shape[3]
        pn = spec.param or spec.name
        w = G.conv_weight(self.seed, pn, spec.c_out, spec.c_in, spec.k, spec.k, net.layout,
                          net.dtype)
        b = G.conv_bias(self.seed, pn, spec.c_out)
        al = G.prelu_alpha(self.seed, pn, spec.c_out) if spec.act == A.ACT_PRELU else None
        net.params[spec.name] = (w, b, al)
        wd, bd = w.to(self.device), b.to(self.device)
        ald = al.to(self.device) if al is not None else None
        y = self.buffer(spec.name, spec.c_out, spec.oh, spec.ow)
        yu = self.buffer(up_name, spec.c_out, 2 * spec.oh, 2 * spec.ow)
        d = A.ConvDesc(net.batch, spec.h, spec.w, spec.c_in, spec.c_out, spec.k, spec.k,
                       spec.stride, spec.pad, net.layout, net.dtype)
        ws_bytes = A.acnn_conv2d_workspace_size(d)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=self.device) if ws_bytes else None
        net.tensors[spec.name + ".ws"] = ws
        net.conv_inputs[spec.name] = (src_a, src_b) if src_b else src_a
        res = net.tensors[residual] if residual else None
        res_mode = spec.res_mode if residual else A.RES_NONE
        if residual:
            net.conv_residuals[spec.name] = residual
        net.upsampled[up_name] = spec.name

        def fn(stream):
            A.check(A.acnn_conv2d_fused_up2(d, xa, ca, xb, wd, bd, ald, res, res_mode, spec.act,
                                            y, yu, ws, ws_bytes, stream), spec.name)

        byts = (xa.numel() + (xb.numel() if xb is not None else 0) + w.numel() + y.numel() +
                yu.numel() + (y.numel() if res is not None else 0)) * self.es + 4 * spec.c_out
        net.ops.append(Op("conv", self.section, fn, _conv_flops(net.batch, spec), byts, spec.name,
                          spec))
        return spec.name

    def conv_cat(self, src_a, src_b, spec: ConvSpec, residual=None, up2=None):
        """spec over the channel concat [src_a | src_b] (NHWC), the concat folded
        into the conv's operand loads (acnn_conv2d_fused_cat2); up2: also write
        the nearest 2x upsample of the output under that name."""
        if up2:
            return self._conv_up2(src_a, src_b, spec, residual, up2)
        net = self.net
        xa, xb = net.tensors[src_a], net.tensors[src_b]
        ca = xa.shape[3]
        w = G.conv_weight(self.seed, spec.name, spec.c_out, spec.c_in, spec.k, spec.k,
                          net.layout, net.dtype)
        b = G.conv_bias(self.seed, spec.name, spec.c_out)
        al = G.prelu_alpha(self.seed, spec.name, spec.c_out) if spec.act == A.ACT_PRELU else None
        net.params[spec.name] = (w, b, al)
        wd, bd = w.to(self.device), b.to(self.device)
        ald = al.to(self.device) if al is not None else None
        y = self.buffer(spec.name, spec.c_out, spec.oh, spec.ow)
        d = A.ConvDesc(net.batch, spec.h, spec.w, spec.c_in, spec.c_out, spec.k, spec.k,
                       spec.stride, spec.pad, net.layout, net.dtype)
        ws_bytes = A.acnn_conv2d_workspace_size(d)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=self.device) if ws_bytes else None
        net.tensors[spec.name + ".ws"] = ws
        net.conv_inputs[spec.name] = (src_a, src_b)
        res = net.tensors[residual] if residual else None
        res_mode = spec.res_mode if residual else A.RES_NONE
        if residual:
            net.conv_residuals[spec.name] = residual

        def fn(stream):
            A.check(A.acnn_conv2d_fused_cat2(d, xa, ca, xb, wd, bd, ald, res, res_mode,
                                             spec.act, y, ws, ws_bytes, stream), spec.name)

        byts = (xa.numel() + xb.numel() + w.numel() + y.numel() +
                (y.numel() if res is not None else 0)) * self.es + 4 * spec.c_out
        net.ops.append(Op("conv", self.section, fn, _conv_flops(net.batch, spec), byts, spec.name,
                          spec))
        return spec.name

    def pool(self, src, dst, kind, k, s, p, c, h, w):
        net = self.net
        x = net.tensors[src]
        oh, ow = (h + 2 * p - k) // s + 1, (w + 2 * p - k) // s + 1
        y = self.buffer(dst, c, oh, ow)
        n = net.batch

        def fn(stream):
            A.check(A.acnn_pool2d(kind, n, h, w, c, k, s, p, net.layout, net.dtype, x, y, stream),
                    dst)

        net.ops.append(Op("pool", self.section, fn, 0.0, (x.numel() + y.numel()) * self.es, dst))
        return dst

    def resize(self, src, dst, mode, c, h, w, oh, ow, out_dtype=None, touched_in=None):
        net = self.net
        x = net.tensors[src]
        od = net.dtype if out_dtype is None else out_dtype
        y = self.buffer(dst, c, oh, ow, dtype=od)
        n = net.batch
        in_dt = A.dtype_code(x.dtype)

        def fn(stream):
            A.check(A.acnn_resize2d(mode, n, c, h, w, oh, ow, net.layout, in_dt, od, x, y, stream),
                    dst)

        rd = touched_in if touched_in is not None else x.numel() * x.element_size()
        net.ops.append(Op("resize", self.section, fn, 0.0, rd + y.numel() * y.element_size(), dst))
        return dst

    def concat(self, a, b, dst, ca, cb, h, w):
        net = self.net
        ta, tb = net.tensors[a], net.tensors[b]
        y = self.buffer(dst, ca + cb, h, w)
        n = net.batch

        def fn(stream):
            A.check(A.acnn_concat(n, h, w, ca, cb, net.layout, net.dtype, ta, tb, y, stream), dst)

        net.ops.append(Op("concat", self.section, fn, 0.0, 2 * y.numel() * self.es, dst))
        return dst


# ============================================================== workloads
def conv1_net(device="cuda") -> Net:
    """Single conv3x3/s1/p1 16->32 + bias + ReLU, NHWC fp32, 1x32x32x16, x ~ U(-1, 1)."""
    seed = 1234
    net = Net("conv1", 1, G.F32, G.NHWC)
    b = Builder(net, seed, device)
    b.set_section("conv")
    x = G.tensor(seed, "x", (1, 32, 32, 16), "uniform", -1.0, 1.0, dtype=G.F32)
    net.tensors["x"] = x.to(device)
    net.inputs["x"] = net.tensors["x"]
    b.conv("x", ConvSpec("conv", 16, 32, 3, 1, 1, A.ACT_RELU, 32, 32))
    net.outputs = ["conv"]
    return net


def stem_specs(h, w, prefix="stem"):
    s0 = ConvSpec(f"{prefix}.0", 3, 32, 3, 2, 1, A.ACT_RELU, h, w)
    s1 = ConvSpec(f"{prefix}.1", 32, 32, 3, 1, 1, A.ACT_RELU, s0.oh, s0.ow)
    s2 = ConvSpec(f"{prefix}.2", 32, 64, 3, 1, 1, A.ACT_RELU, s1.oh, s1.ow)
    return [s0, s1, s2]


def _stem(b: Builder, src, h, w):
    specs = stem_specs(h, w)
    cur = src
    for s in specs:
        cur = b.conv(cur, s)
    s2 = specs[-1]
    return b.pool(cur, "stem.pool", A.POOL_MAX, 3, 2, 1, 64, s2.oh, s2.ow), \
        (s2.oh + 2 - 3) // 2 + 1, (s2.ow + 2 - 3) // 2 + 1


def stem_net(device="cuda", n=1, h=640, w=640) -> Net:
    """ResNet-D stem, NHWC fp32: 3 convs (+ReLU) then maxpool 3/2/1; x ~ U(0, 1)."""
    seed = 1235
    net = Net("stem", n, G.F32, G.NHWC)
    b = Builder(net, seed, device)
    b.set_section("stem")
    x = G.tensor(seed, "x", (n, h, w, 3), "uniform", 0.0, 1.0, dtype=G.F32)
    net.tensors["x"] = x.to(device)
    net.inputs["x"] = net.tensors["x"]
    out, _, _ = _stem(b, "x", h, w)
    net.outputs = [out]
    return net


def bottleneck(b: Builder, src, name, c_in, width, h, w, stride, shortcut, pooled=None,
               pool_out=False):
    """ResNet-D bottleneck: 1x1 -> 3x3 (stride here) -> 1x1, shortcut, add, ReLU.

    shortcut: 'identity', 'conv' (1x1, stride 1) or 'pool' (avgpool 2x2/s2 then 1x1).
    The add and the ReLU run in the last conv's epilogue (residual before act).
    pooled: the name of src's 2x2/s2 average pool when the previous block's last
    conv already wrote it (the 'pool' shortcut then runs no pool of its own);
    pool_out: this block's last conv also writes the average pool of its output
    (tensor f"{name}.pooled"), for the next stage's shortcut.
    """
    mid = width // 4
    c1 = ConvSpec(f"{name}.conv1", c_in, mid, 1, 1, 0, A.ACT_RELU, h, w)
    c2 = ConvSpec(f"{name}.conv2", mid, mid, 3, stride, 1, A.ACT_RELU, h, w)
    c3 = ConvSpec(f"{name}.conv3", mid, width, 1, 1, 0, A.ACT_RELU, c2.oh, c2.ow,
                  res_mode=A.RES_ADD_THEN_ACT)
    # the shortcut branch runs beside conv1 -> conv2 (a parallel branch of the
    # section's graph: these layers leave SMs idle), joined before conv3
    if shortcut == "identity":
        res = src
    else:
        with b.side():
            if shortcut == "conv":
                res = b.conv(src, ConvSpec(f"{name}.short", c_in, width, 1, 1, 0, A.ACT_NONE,
                                           h, w))
            else:
                if pooled is None:
                    pooled = b.pool(src, f"{name}.pool", A.POOL_AVG, 2, 2, 0, c_in, h, w)
                res = b.conv(pooled, ConvSpec(f"{name}.short", c_in, width, 1, 1, 0,
                                              A.ACT_NONE, h // 2, w // 2))
    t = b.conv(src, c1)
    t = b.conv(t, c2)
    out = b.conv(t, c3, residual=res, pool2=f"{name}.pooled" if pool_out else None)
    b.net.ops[-1].join = True
    return out, c2.oh, c2.ow


def block_net(device="cuda", variant="identity", n=4, h=80, w=80) -> Net:
    """Bottleneck at 4x80x80x256, NHWC bf16, x ~ N(0, 1): identity or downsample variant."""
    seed = 1236
    net = Net(f"block_{variant}", n, G.BF16, G.NHWC)
    b = Builder(net, seed, device)
    b.set_section(variant)
    x = G.tensor(seed, "x", (n, h, w, 256), "normal", dtype=G.BF16)
    net.tensors["x"] = x.to(device)
    net.inputs["x"] = net.tensors["x"]
    if variant == "identity":
        out, _, _ = bottleneck(b, "x", "id", 256, 256, h, w, 1, "identity")
    else:
        out, _, _ = bottleneck(b, "x", "down", 256, 512, h, w, 2, "pool")
    net.outputs = [out]
    return net


STAGES = [(3, 256, 1, "conv"), (4, 512, 2, "pool"), (6, 1024, 2, "pool"), (3, 2048, 2, "pool")]


def csp_block(b: Builder, src_a, src_b, name, h, w, blocks=3, hidden=256, up2=None):
    """CSP block over [src_a | src_b] (512 channels) -> 256, as P1
    RtDetrGpu::csp composes it: a = conv1(x); per RepVGG bottleneck
    a = SiLU(conv3x3(a) + conv1x1(a)); out = a + conv2(x).  conv1 and conv2 are
    1x1 + SiLU reading the concat folded into their operand loads; the RepVGG
    sum is the 3x3 conv's add-then-activate residual (the 1x1's output, no
    activation); the final add is conv2's activate-then-add residual."""
    S = A.ACT_SILU
    a = b.conv_cat(src_a, src_b, ConvSpec(f"{name}.conv1", 512, hidden, 1, 1, 0, S, h, w))
    for i in range(blocks):
        q = b.conv(a, ConvSpec(f"{name}.rep{i}.conv1x1", hidden, hidden, 1, 1, 0, A.ACT_NONE, h, w))
        a = b.conv(a, ConvSpec(f"{name}.rep{i}.conv3x3", hidden, hidden, 3, 1, 1, S, h, w,
                               res_mode=A.RES_ADD_THEN_ACT), residual=q)
    return b.conv_cat(src_a, src_b, ConvSpec(name, 512, 256, 1, 1, 0, S, h, w,
                                             res_mode=A.RES_ACT_THEN_ADD), residual=a, up2=up2)


def backbone_net(device="cuda", n=8, h=640, w=640, neck="fusion") -> Net:
    """ResNet-D-50 backbone + neck, NHWC bf16, N x 640 x 640 x 3, x ~ U(0, 1).

    Neck (top-down then bottom-up, every conv + SiLU): lateral 1x1 convs to 256
    on C3/C4/C5; F5 = lat5; F4 = conv3x3(cat[up2(F5), lat4]);
    F3 = conv3x3(cat[up2(F4), lat3]); N4 = conv3x3(cat[conv3x3/s2(F3), F4]);
    N5 = conv3x3(cat[conv3x3/s2(N4), F5]).  Outputs F3, N4, N5.  Each concat is
    folded into the conv that reads it (acnn_conv2d_fused_cat2: the conv's
    operand loads take channels 0-255 from one map and 256-511 from the other).
    neck="csp": each of the four 3x3 fusion convs becomes a CSP block with three
    RepVGG bottlenecks (csp_block), as P1's neck has them.
    """
    seed = 1238
    net = Net("backbone" if neck == "fusion" else "backbone_csp", n, G.BF16, G.NHWC)
    b = Builder(net, seed, device)
    x = G.tensor(seed, "x", (n, h, w, 3), "uniform", 0.0, 1.0, dtype=G.BF16)
    net.tensors["x"] = x.to(device)
    net.inputs["x"] = net.tensors["x"]
    b.set_section("stem")
    cur, ch, cw = _stem(b, "x", h, w)
    c_in = 64
    feats = []
    pooled = None
    for si, (blocks, width, stride, first_short) in enumerate(STAGES):
        b.set_section(f"stage{si + 1}")
        for bi in range(blocks):
            short = first_short if bi == 0 else "identity"
            # a stage's last block also writes the average pool of its output
            # when the next stage's shortcut pools it (cross-op fusion)
            pool_out = (bi == blocks - 1 and si + 1 < len(STAGES) and STAGES[si + 1][3] == "pool"
                        and ch % 2 == 0 and cw % 2 == 0)
            name = f"s{si + 1}.b{bi}"
            cur, ch, cw = bottleneck(b, cur, name, c_in, width, ch, cw,
                                     stride if bi == 0 else 1, short,
                                     pooled=pooled if bi == 0 else None, pool_out=pool_out)
            pooled = f"{name}.pooled" if pool_out else None
            c_in = width
        feats.append((cur, ch, cw, width))
    b.set_section("neck")
    (c3, h3, w3, ch3), (c4, h4, w4, ch4), (c5, h5, w5, ch5) = feats[1], feats[2], feats[3]
    S = A.ACT_SILU
    # lat3 and lat4 run beside lat5 (parallel branch), joined before the first
    # fusion conv that reads them
    with b.side():
        lat3 = b.conv(c3, ConvSpec("neck.lat3", ch3, 256, 1, 1, 0, S, h3, w3))
        lat4 = b.conv(c4, ConvSpec("neck.lat4", ch4, 256, 1, 1, 0, S, h4, w4))

    def fuse(src_a, src_b, name, hh, ww, up2=None):
        if neck == "csp":
            return csp_block(b, src_a, src_b, name, hh, ww, up2=up2)
        return b.conv_cat(src_a, src_b, ConvSpec(name, 512, 256, 3, 1, 1, S, hh, ww), up2=up2)

    # the two top-down nearest 2x upsamples are written by the convs that
    # produce the maps they upsample (cross-op fusion), when the sizes double
    fold = 2 * h5 == h4 and 2 * w5 == w4 and 2 * h4 == h3 and 2 * w4 == w3
    if fold:
        f5 = b.conv(c5, ConvSpec("neck.lat5", ch5, 256, 1, 1, 0, S, h5, w5), up2="neck.up5")
        up5 = "neck.up5"
        first = len(net.ops)
        f4 = fuse(up5, lat4, "neck.fpn4", h4, w4, up2="neck.up4")
        up4 = "neck.up4"
    else:
        f5 = b.conv(c5, ConvSpec("neck.lat5", ch5, 256, 1, 1, 0, S, h5, w5))
        up5 = b.resize(f5, "neck.up5", A.RESIZE_NEAREST, 256, h5, w5, h4, w4)
        first = len(net.ops)
        f4 = fuse(up5, lat4, "neck.fpn4", h4, w4)
        up4 = b.resize(f4, "neck.up4", A.RESIZE_NEAREST, 256, h4, w4, h3, w3)
    net.ops[first].join = True
    f3 = fuse(up4, lat3, "neck.fpn3", h3, w3)
    d3 = b.conv(f3, ConvSpec("neck.down3", 256, 256, 3, 2, 1, S, h3, w3))
    n4 = fuse(d3, f4, "neck.pan4", h4, w4)
    d4 = b.conv(n4, ConvSpec("neck.down4", 256, 256, 3, 2, 1, S, h4, w4))
    n5 = fuse(d4, f5, "neck.pan5", h5, w5)
    net.outputs = [f3, n4, n5]
    return net


def frame_net(device="cuda", h=1088, w=1920, c1=120, c2=240, t=0.5, flow_out=False) -> Net:
    """Frame-interpolation conv stack, NCHW fp16 (rt.js run(), first 13 dispatches).

    prep (bilinear 1/4 of both RGBA8 frames + t plane) -> conv3x3/s2 7->c1 + PReLU
    -> conv3x3/s2 c1->c2 + PReLU -> 8 x conv3x3 c2->c2 + PReLU, the 8th adding the
    map that entered the 8 (after its PReLU) -> deconv 4x4/s2 c2->5 -> bilinear x8;
    with flow_out, the last step is instead the flow-out stage (x8 upsample, warp
    of both frames, blend, RGBA8 output frame).
    """
    seed = 1237
    net = Net("frame_out" if flow_out else "frame", 1, G.F16, G.NCHW)
    b = Builder(net, seed, device)
    b.set_section("frame")
    f0 = G.rgba_frame(seed, "frame0", h, w).to(device)
    f1 = G.rgba_frame(seed, "frame1", h, w).to(device)
    net.tensors["frame0"], net.tensors["frame1"] = f0, f1
    net.inputs["frame0"], net.inputs["frame1"] = f0, f1
    qh, qw = h // 4, w // 4
    xq = b.buffer("xq", 7, qh, qw)

    def prep(stream):
        A.check(A.acnn_frame_prep_quarter(h, w, f0, f1, t, G.F16, xq, stream), "prep")

    touched = 2 * (2 * qh) * w * 4  # two source rows per output row, both frames
    net.ops.append(Op("prep", "frame", prep, 0.0, touched + xq.numel() * 2, "prep"))
    P = A.ACT_PRELU
    # each conv of the chain writes an NHWC copy of its output for the next
    # (rt.js keeps one layout throughout; here the NCHW maps stay as stored
    # and the tensor-core convs read the copies instead of staging)
    a = b.conv("xq", ConvSpec("conv0a", 7, c1, 3, 2, 1, P, qh, qw), nhwc_copy=True)
    s0 = ConvSpec("conv0b", c1, c2, 3, 2, 1, P, qh // 2, qw // 2)
    cur = b.conv(a, s0, nhwc_copy=True)
    skip = cur
    hh, ww = s0.oh, s0.ow
    for i in range(8):
        last = i == 7
        spec = ConvSpec(f"convblock.{i}", c2, c2, 3, 1, 1, P, hh, ww,
                        res_mode=A.RES_ACT_THEN_ADD if last else A.RES_NONE)
        cur = b.conv(cur, spec, residual=skip if last else None, nhwc_copy=not last)
    wdc = G.deconv_weight(seed, "lastconv", c2, 5, 4)
    bdc = G.conv_bias(seed, "lastconv", 5)
    net.params["lastconv"] = (wdc, bdc, None)
    wdd, bdd = wdc.to(device), bdc.to(device)
    xin = net.tensors[cur]
    tmp8 = b.buffer("tmp8", 5, 2 * hh, 2 * ww)
    dd = A.ConvDesc(1, hh, ww, c2, 5, 4, 4, 2, 1, G.NCHW, G.F16)

    def deconv(stream):
        A.check(A.acnn_deconv2d(dd, xin, wdd, bdd, None, A.ACT_NONE, G.F16, tmp8, stream),
                "deconv")

    net.ops.append(Op("deconv", "frame", deconv, 2.0 * 5 * c2 * 4 * (2 * hh) * (2 * ww),
                      (xin.numel() + tmp8.numel()) * 2 + wdc.numel() * 4, "deconv"))
    if not flow_out:
        b.resize("tmp8", "flow", A.RESIZE_BILINEAR, 5, 2 * hh, 2 * ww, h, w)
        net.outputs = ["flow"]
        return net
    # flow-out stage (rt.js wgslFlowOut): x8 upsample of tmp8, warp both
    # frames by their flows, sigmoid-mask blend, RGBA8 pack
    out = torch.empty((h, w, 4), dtype=torch.uint8, device=device)
    net.tensors["out"] = out

    def flow_stage(stream):
        A.check(A.acnn_frame_flow_out(h, w, tmp8, G.F16, f0, f1, None, out, stream), "flow_out")

    # algorithmic bytes: the 1/8 map, both frames once, the output frame
    net.ops.append(Op("flow_out", "frame", flow_stage, 0.0,
                      tmp8.numel() * 2 + 3 * h * w * 4, "flow_out"))
    net.outputs = ["out"]
    return net


def frame_tfact_net(device="cuda", h=1088, w=1920, c1=120, c2=240, ts=(0.25, 0.5, 0.75),
                    hn=64, rc=32) -> Net:
    """t-factored frame stack with the refine head (rt.js tfact2: prepPair once
    per frame pair, runT per timestep), NCHW fp16.

    trunk, once: prep (the six frame planes of the bilinear 1/4 prep) -> conv3x3/s2
    6->c1 + PReLU -> conv3x3/s2 c1->c2 + PReLU (feat0) -> convblocks 0..5.
    per t: FiLM(t) of the trunk map -> convblocks 6, 7 (7 adds feat0 after its
    PReLU) -> deconv 4x4/s2 c2->5 -> refine prep (11 planes at 1/4) -> three
    conv3x3 + PReLU (11->rc->rc->rc, zero padding) -> refine out (replicate-padded
    conv3x3 rc->3, 2 sigmoid - 1, fp32) -> flow-out with that residual.
    Outputs: one h x w RGBA8 frame per t.
    """
    assert rc % 4 == 0, "refine channels must be a multiple of 4"
    seed = 1238
    net = Net("frame_tfact", 1, G.F16, G.NCHW)
    b = Builder(net, seed, device)
    b.set_section("frame")
    f0 = G.rgba_frame(seed, "frame0", h, w).to(device)
    f1 = G.rgba_frame(seed, "frame1", h, w).to(device)
    net.tensors["frame0"], net.tensors["frame1"] = f0, f1
    net.inputs["frame0"], net.inputs["frame1"] = f0, f1
    qh, qw = h // 4, w // 4
    # the 6-channel prep is the first six planes of the 7-plane prep (its t
    # plane is written and not read): the same kernel, no second variant
    xq = b.buffer("xq", 7, qh, qw)
    net.tensors["xq6"] = xq[:, :6]

    def prep(stream):
        A.check(A.acnn_frame_prep_quarter(h, w, f0, f1, 0.0, G.F16, xq, stream), "prep")

    touched = 2 * (2 * qh) * w * 4
    net.ops.append(Op("prep", "frame", prep, 0.0, touched + xq.numel() * 2, "prep"))
    P = A.ACT_PRELU
    a = b.conv("xq6", ConvSpec("conv0a", 6, c1, 3, 2, 1, P, qh, qw), nhwc_copy=True)
    s0 = ConvSpec("conv0b", c1, c2, 3, 2, 1, P, qh // 2, qw // 2)
    feat0 = b.conv(a, s0, nhwc_copy=True)
    hh, ww = s0.oh, s0.ow
    cur = feat0
    for i in range(6):
        cur = b.conv(cur, ConvSpec(f"convblock.{i}", c2, c2, 3, 1, 1, P, hh, ww),
                     nhwc_copy=i < 5)  # the trunk's last map feeds FiLM (NCHW)
    trunk = net.tensors[cur]
    fw = [t.to(device) for t in G.film_mlp(seed, "film", c2, hn)]
    net.params["film"] = G.film_mlp(seed, "film", c2, hn)
    wdc = G.deconv_weight(seed, "lastconv", c2, 5, 4)
    bdc = G.conv_bias(seed, "lastconv", 5)
    net.params["lastconv"] = (wdc, bdc, None)
    wdd, bdd = wdc.to(device), bdc.to(device)
    wro = G.refine_out_weight(seed, "refine.c3", rc)
    bro = G.conv_bias(seed, "refine.c3", 3)
    net.params["refine.c3"] = (wro, bro, None)
    wrod, brod = wro.to(device), bro.to(device)
    dd = A.ConvDesc(1, hh, ww, c2, 5, 4, 4, 2, 1, G.NCHW, G.F16)
    outs = []
    for i, t in enumerate(ts):
        sfx = f"@t{i}"
        fm = b.buffer("film" + sfx, c2, hh, ww)

        def film(stream, t=t, fm=fm):
            A.check(A.acnn_film(c2, hh * ww, G.F16, trunk, t, *fw[:2], hn, *fw[2:], fm, stream),
                    "film")

        net.ops.append(Op("film", "frame", film, 2.0 * c2 * hh * ww + 4.0 * c2 * hn,
                          2 * trunk.numel() * 2, "film" + sfx))
        cur = b.conv("film" + sfx, ConvSpec("convblock.6" + sfx, c2, c2, 3, 1, 1, P, hh, ww,
                                            param="convblock.6"), nhwc_copy=True)
        cur = b.conv(cur, ConvSpec("convblock.7" + sfx, c2, c2, 3, 1, 1, P, hh, ww,
                                   res_mode=A.RES_ACT_THEN_ADD, param="convblock.7"),
                     residual=feat0)
        xin = net.tensors[cur]
        tmp8 = b.buffer("tmp8" + sfx, 5, 2 * hh, 2 * ww)

        def deconv(stream, xin=xin, tmp8=tmp8):
            A.check(A.acnn_deconv2d(dd, xin, wdd, bdd, None, A.ACT_NONE, G.F16, tmp8, stream),
                    "deconv")

        net.ops.append(Op("deconv", "frame", deconv, 2.0 * 5 * c2 * 4 * (2 * hh) * (2 * ww),
                          (xin.numel() + tmp8.numel()) * 2 + wdc.numel() * 4, "deconv" + sfx))
        rin = b.buffer("rin" + sfx, 11, qh, qw)

        def rprep(stream, tmp8=tmp8, rin=rin):
            A.check(A.acnn_frame_refine_prep(h, w, tmp8, G.F16, f0, f1, G.F16, rin, stream),
                    "refine_prep")

        # algorithmic bytes: the 1/8 map, the frames' pixels the four centre taps
        # of each 4x4 block reach (about half of each frame), the 11 planes
        net.ops.append(Op("refine_prep", "frame", rprep, 0.0,
                          tmp8.numel() * 2 + 2 * (h * w * 4) // 2 + rin.numel() * 2,
                          "refine_prep" + sfx))
        r = b.conv("rin" + sfx, ConvSpec("refine.c0" + sfx, 11, rc, 3, 1, 1, P, qh, qw,
                                         param="refine.c0"), nhwc_copy=True)
        r = b.conv(r, ConvSpec("refine.c1" + sfx, rc, rc, 3, 1, 1, P, qh, qw, param="refine.c1"),
                   nhwc_copy=True)
        r = b.conv(r, ConvSpec("refine.c2" + sfx, rc, rc, 3, 1, 1, P, qh, qw, param="refine.c2"))
        rx = net.tensors[r]
        rres = b.buffer("rres" + sfx, 3, qh, qw, dtype=G.F32)

        def rout(stream, rx=rx, rres=rres):
            A.check(A.acnn_frame_refine_out(rc, qh, qw, rx, G.F16, wrod, brod, rres, stream),
                    "refine_out")

        net.ops.append(Op("refine_out", "frame", rout, 2.0 * 3 * rc * 9 * qh * qw,
                          rx.numel() * 2 + rres.numel() * 4, "refine_out" + sfx))
        out = torch.empty((h, w, 4), dtype=torch.uint8, device=device)
        net.tensors["out" + sfx] = out

        def flow_stage(stream, tmp8=tmp8, rres=rres, out=out):
            A.check(A.acnn_frame_flow_out(h, w, tmp8, G.F16, f0, f1, rres, out, stream),
                    "flow_out")

        net.ops.append(Op("flow_out", "frame", flow_stage, 0.0,
                          tmp8.numel() * 2 + rres.numel() * 4 + 3 * h * w * 4,
                          "flow_out" + sfx))
        outs.append("out" + sfx)
    net.outputs = outs
    return net


WORKLOADS = {
    "conv1": conv1_net,
    "stem": stem_net,
    "block": lambda device="cuda": block_net(device, "identity"),
    "block_down": lambda device="cuda": block_net(device, "downsample"),
    "frame": frame_net,
    "frame_out": lambda device="cuda": frame_net(device, flow_out=True),
    "backbone": backbone_net,
    "backbone_csp": lambda device="cuda": backbone_net(device, neck="csp"),
    "frame_tfact": frame_tfact_net,
}
