"""Tile sweep of the tensor-core conv: every instantiated plan of every conv of
a workload, timed on the device, against the planner's own choice.

The offline form of rt.js's one-shot conv autotune (tuneConvRB, which times
its register-blocked variants once on the adapter and keeps the fastest):
each tensor-core conv layer of the workload is run alone with each tile shape
(output channels x output pixels per tile) and K split the kernel has, forced
through acnn_conv2d_force_plan, as a one-launch CUDA graph replayed after an
L2 flush (CUDA events on the launching stream).  Inputs are seeded random
tensors of the layer's shapes; a channel concat folded into a conv is swept as
the plain conv over the concatenated channels (the same GEMM).

    python -m activation_cnn_gb300.tune [--workload backbone] [--reps 20]

prints one JSON object: per layer the planner's plan and time, the fastest
plan and time, and every plan tried.
"""
from __future__ import annotations

import argparse
import json
import statistics

import torch

from . import acnn as A
from . import inputs as G
from . import network as N

L2_FLUSH_BYTES = 512 << 20
# (output channels, output pixels) per tile with a kernel instantiation, by
# channels per k-block (64, or 32 when C_in <= 32)
SHAPES = {64: [(256, 128), (128, 128), (128, 256), (64, 128), (64, 256)],
          32: [(128, 256), (64, 256), (32, 256)]}
SPLITS = (1, 2, 3, 4, 6, 8)


def _time(fn, stream, flush, reps):
    """Median device time of fn() captured in a graph, L2 flushed before each replay."""
    sec = A.Section(stream)
    with torch.cuda.stream(stream):
        fn(stream)  # once eagerly (checks the call)
    stream.synchronize()
    with torch.cuda.stream(stream):
        with sec:
            fn(stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for _ in range(reps):
        flush()
        e0.record(stream)
        sec.launch(stream)
        e1.record(stream)
        stream.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e-3)
    sec.close()
    st = A.acnn_last_device_status(stream.cuda_stream)
    if st != 0:
        raise RuntimeError(f"device status {A.status_string(st)}")
    return statistics.median(ts)


def sweep_layer(spec, net, stream, flush, reps, seed=77):
    n, layout, dtype = net.batch, net.layout, net.dtype
    d = A.ConvDesc(n, spec.h, spec.w, spec.c_in, spec.c_out, spec.k, spec.k, spec.stride,
                   spec.pad, layout, dtype)
    if A.acnn_conv2d_path(d) not in (1, 2):
        return None
    dev = stream.device
    x = G.tensor(seed, spec.name + ".tx", G.activation_shape(layout, n, spec.c_in, spec.h, spec.w),
                 "normal", dtype=dtype).to(dev)
    w = G.conv_weight(seed, spec.name + ".t", spec.c_out, spec.c_in, spec.k, spec.k, layout,
                      dtype).to(dev)
    b = G.conv_bias(seed, spec.name + ".t", spec.c_out).to(dev)
    al = G.prelu_alpha(seed, spec.name + ".t", spec.c_out).to(dev)
    ys = G.activation_shape(layout, n, spec.c_out, spec.oh, spec.ow)
    y = torch.empty(ys, dtype=G.TORCH_DTYPE[dtype], device=dev)
    res = torch.randn(ys, device=dev).to(y.dtype) if spec.res_mode else None

    def run_plan():
        ws_bytes = A.acnn_conv2d_workspace_size(d)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        st, rows, bn, splits = A.acnn_conv2d_plan(d, ws_bytes)
        assert st == 0

        def fn(s):
            A.check(A.acnn_conv2d_fused(d, x, w, b, al, res, spec.res_mode if res is not None
                                        else A.RES_NONE, spec.act, y, ws, ws_bytes, s),
                    spec.name)
        return (bn, rows, splits), _time(fn, stream, flush, reps)

    A.acnn_conv2d_force_plan(0)
    default, t_default = run_plan()
    tried = {default: t_default}
    bk = 32 if spec.c_in <= 32 else 64
    for bn, rows in SHAPES[bk]:
        if bn > 2 * max(32, spec.c_out):
            continue
        for sp in SPLITS if layout == G.NHWC else (1,):
            A.acnn_conv2d_force_plan(bn, rows, sp)
            st, r2, b2, s2 = A.acnn_conv2d_plan(d, A.acnn_conv2d_workspace_size(d))
            if (b2, r2, s2) in tried:
                continue
            plan, t = run_plan()
            tried[plan] = t
    A.acnn_conv2d_force_plan(0)
    best = min(tried, key=tried.get)
    flops = 2.0 * n * spec.oh * spec.ow * spec.c_out * spec.c_in * spec.k * spec.k
    return {"name": spec.name, "geometry": [n, spec.h, spec.w, spec.c_in, spec.c_out, spec.k,
                                            spec.stride],
            "default": {"bn_rows_splits": list(default), "us": round(t_default * 1e6, 2)},
            "best": {"bn_rows_splits": list(best), "us": round(tried[best] * 1e6, 2)},
            "best_TFLOP_s": round(flops / tried[best] / 1e12, 1),
            "all": [{"bn_rows_splits": list(k), "us": round(v * 1e6, 2)}
                    for k, v in sorted(tried.items(), key=lambda kv: kv[1])]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="backbone")
    ap.add_argument("--reps", type=int, default=20)
    args = ap.parse_args()
    from . import build as B
    B.build()
    A.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    net = N.WORKLOADS[args.workload](dev)
    stream = torch.cuda.Stream(device=dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush():
        with torch.cuda.stream(stream):
            flush_buf.add_(1)

    out, seen = [], set()
    for op in net.ops:
        if op.kind != "conv" or op.spec is None:
            continue
        s = op.spec
        key = (s.h, s.w, s.c_in, s.c_out, s.k, s.stride, s.pad, s.act, s.res_mode)
        if key in seen:  # identical layers (repeated blocks) are swept once
            continue
        seen.add(key)
        r = sweep_layer(s, net, stream, flush, args.reps)
        if r is not None:
            out.append(r)
    tot_d = sum(r["default"]["us"] for r in out)
    tot_b = sum(r["best"]["us"] for r in out)
    print(json.dumps({"workload": args.workload, "layers": out,
                      "sum_default_us": round(tot_d, 1), "sum_best_us": round(tot_b, 1)}))


if __name__ == "__main__":
    main()
