"""Benchmark: backbone+neck images/s (and fused-conv TFLOP/s) on GB300.

python bench.py [--gpus N --steps K --warmup W] [--workload backbone|block|...]
               [--impl ours|reference] [--no-cpu-baseline]

A step is one pass of the whole workload (every op of every section) over one
batch of synthetic input already resident in HBM: the default workload is the
ResNet-D-50 backbone + neck at 8 x 640 x 640 x 3, NHWC bf16.  Each step replays
the workload's per-section CUDA graphs; L2 is flushed (a 512 MB write) before
every step, outside the timed interval.  Under torchrun each rank runs its own
batch (weak scaling, replicas: no data-path collective); the reported time is
the max over ranks.

Printed: ONE JSON line on rank 0 with value (img/s), the fused-conv TFLOP/s,
a roofline object for the dominant kernel (the tcgen05 implicit-GEMM conv,
per-launch times from CUDA events recorded inside the graphs), an
end-to-end figure through host buffers, the oracle timed on the host cores,
the SM clocks sampled during the timed region and the kernel launch count.

--impl reference times the fp64 CPU oracle on the same workload and metric
(each step a bounded sample), rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("fused-conv TFLOP/s (% of GB300 BF16 dense peak); backbone img/s @640x640")
L2_BYTES = 129 << 20  # GB300 L2
L2_FLUSH_BYTES = 512 << 20


def kernel_source_hash():
    """sha256 of the tensor-core conv source, to tie ncu counters to the kernel they measured."""
    import hashlib
    src = os.path.join(ROOT, "activation_cnn_gb300", "csrc", "conv_igemm.cu")
    with open(src, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


# DRAM traffic of the tensor-core conv kernel, per launch, averaged over the
# conv launches of one backbone step: dram__bytes_read.sum +
# dram__bytes_write.sum from an ncu capture (a one-pass metric pair) of the
# kernel source with this sha256 prefix.  None once the source has changed
# since the counters were taken.
CONV_TRAFFIC = {"kernel_sha16": "a08b83565c22dbdc", "bytes_per_launch": 4 * 10.218e6,
                "how": "ncu dram__bytes_read.sum + dram__bytes_write.sum (one pass) over the 63 "
                       "conv launches of one pass at batch 2, x 4 rows for batch 8; writes that "
                       "stay dirty in L2 through a launch are not attributed to it"}


def conv_traffic(workload, batch):
    """Per-launch DRAM bytes of the conv kernel for the default backbone step,
    or None when they were measured on another version of the kernel."""
    if workload != "backbone" or batch not in (None, 8):
        return None
    if CONV_TRAFFIC["kernel_sha16"] != kernel_source_hash():
        return None
    return CONV_TRAFFIC["bytes_per_launch"]


# FP32 FFMA peak of a GB300 (derived, not measured): 152 SMs x 128 FP32 lanes x
# 2 FLOP per FMA x 2.07 GHz maximum SM clock.
FP32_FFMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"bf16_burst": d.get("bf16_tflops"), "bf16_sustained": d.get("bf16_tflops_sustained"),
                "hbm": d.get("hbm_gbs"), "source": "measured"}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        # the timed region starts only once samples are flowing
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for name, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm
def build_net(name, device, batch=None):
    from activation_cnn_gb300 import network as N
    if name == "backbone":
        return N.backbone_net(device, n=batch or 8)
    if name == "backbone_csp":
        return N.backbone_net(device, n=batch or 8, neck="csp")
    if name == "block":
        return N.block_net(device, "identity", n=batch or 4)
    if name == "block_down":
        return N.block_net(device, "downsample", n=batch or 4)
    return N.WORKLOADS[name](device)


def workload_config(name, net, world):
    from activation_cnn_gb300 import inputs as G
    base = {"workload": name, "batch_per_gpu": net.batch, "global_batch": net.batch * world,
            "dtype": {G.F32: "f32", G.F16: "f16", G.BF16: "bf16"}[net.dtype],
            "layout": "NHWC" if net.layout == G.NHWC else "NCHW",
            "parallelism": f"replicas x{world}", "l2": "flushed (512 MB write) before every step",
            "graphs": "one CUDA graph per section: " + ",".join(net.order)}
    if name == "backbone":
        base.update({"image": "640x640x3", "model": "ResNet-D-50 (3/4/6/3) + top-down/bottom-up neck"})
    if name == "backbone_csp":
        base.update({"image": "640x640x3",
                     "model": "ResNet-D-50 (3/4/6/3) + neck with CSP/RepVGG fusion blocks"})
    return base


def launches_per_step(net):
    """Kernels of this library launched by one pass of the network: each op
    records its own count (a conv is one implicit-GEMM launch -- a K split
    reduces inside it, and the split's counter reset is a memset, not a kernel
    -- plus, for the packed path or an NCHW conv, the activation staging
    kernel; the weights of those are prepacked once when the network is built)."""
    return sum(op.launches for op in net.ops)


def time_ops(net, stream, steps, flush):
    """Per-launch device time of every op, from external events inside the graphs.

    Each op of each section is bracketed by two CUDA events recorded as event
    nodes of the section's graph (on the launching stream); the graphs are
    replayed `steps` times after an L2 flush and the per-op times averaged."""
    import torch
    from activation_cnn_gb300 import acnn as A
    evs = {id(op): (torch.cuda.Event(enable_timing=True, external=True),
                    torch.cuda.Event(enable_timing=True, external=True)) for op in net.ops}
    graphs = []
    for sec in net.order:
        g = A.Section(stream)
        with torch.cuda.stream(stream):
            with g:
                for op in net.ops:
                    if op.section != sec:
                        continue
                    evs[id(op)][0].record(stream)
                    op.fn(stream)
                    evs[id(op)][1].record(stream)
        graphs.append(g)
    per_op = {id(op): [] for op in net.ops}
    for _ in range(steps):
        flush()
        for g in graphs:
            g.launch(stream)
        stream.synchronize()
        for op in net.ops:
            a, b = evs[id(op)]
            per_op[id(op)].append(a.elapsed_time(b) * 1e-3)
    for g in graphs:
        g.close()
    rows = []
    for op in net.ops:
        path = None
        if op.kind == "conv":
            s = op.spec
            d = A.ConvDesc(net.batch, s.h, s.w, s.c_in, s.c_out, s.k, s.k, s.stride, s.pad,
                           net.layout, net.dtype)
            path = A.acnn_conv2d_path(d)
        rows.append({"name": op.label, "kind": op.kind, "path": path, "flops": op.flops,
                     "bytes": op.bytes, "section": op.section,
                     "s": statistics.mean(per_op[id(op)])})
    return rows


def time_sections(net, stream, steps, flush):
    """Device time of each captured section graph replayed alone after an L2
    flush (CUDA events on the launching stream), averaged over `steps`."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = {sec: 0.0 for sec, _ in net.graphs}
    for _ in range(steps):
        for sec, g in net.graphs:
            flush()
            e0.record(stream)
            g.launch(stream)
            e1.record(stream)
            stream.synchronize()
            out[sec] += e0.elapsed_time(e1) * 1e-3
    return {k: v / steps for k, v in out.items()}


def apportion(rows, sections, step_s):
    """Split the measured step time over the ops (key "t", seconds per step).

    Each op gets its section's share of the step (sections replayed alone,
    time_sections) times its own share of that section's per-op event time
    (time_ops).  The per-op times, bracketed by event nodes, serialise the
    launches and so overstate every op by its launch gap; the step and the
    sections keep the overlap of consecutive launches.  The apportioned times
    sum to the step, so no op is credited with more time than the step has."""
    tot_sec = sum(sections.values())
    by_sec = {}
    for r in rows:
        by_sec[r["section"]] = by_sec.get(r["section"], 0.0) + r["s"]
    for r in rows:
        r["t"] = step_s * (sections[r["section"]] / tot_sec) * (r["s"] / by_sec[r["section"]])
    return rows


def op_summary(r, pk):
    """One op's apportioned time, throughput and fraction of its roof."""
    t = r["t"]
    d = {"name": r["name"], "kind": r["kind"], "us": round(t * 1e6, 2)}
    if r["flops"]:
        d["TFLOP_s"] = round(r["flops"] / t / 1e12, 2)
    if r["bytes"]:
        d["GB_s"] = round(r["bytes"] / t / 1e9, 1)
    if r["kind"] == "conv":
        d["path"] = r["path"]
        if r["path"] == 0:
            d["frac_fp32_ffma"] = round(r["flops"] / t / 1e12 / FP32_FFMA_TFLOPS, 4)
        else:
            d["frac_tensor_peak"] = round(r["flops"] / t / 1e12 / pk["bf16_burst"], 4)
            roof = max(r["flops"] / (pk["bf16_burst"] * 1e12), r["bytes"] / (pk["hbm"] * 1e9))
            d["attainable_frac"] = round(roof / t, 4)
    elif r["bytes"]:
        d["frac_hbm"] = round(r["bytes"] / t / 1e9 / pk["hbm"], 4)
    return d


def time_steps(net, stream, steps, flush):
    """Device time of `steps` whole steps (every section graph), L2 flushed
    before each step outside the timed interval; returns seconds per step."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush()
        starts[i].record(stream)
        net.replay(stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e-3 for a, b in zip(starts, ends)]


def time_call(fn, stream, flush, reps):
    """Median device time of fn(stream) captured as a graph, L2 flushed before each replay."""
    import torch
    from activation_cnn_gb300 import acnn as A
    with torch.cuda.stream(stream):
        fn(stream)
    stream.synchronize()
    sec = A.Section(stream)
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
    return statistics.median(ts)


def tiny_cin_compare(dev, stream, flush, reps=30):
    """The convs with 3 or 7 input channels (the backbone's RGB stem, the frame
    stack's first conv) on each kernel that serves them: the packed tensor-core
    path the router uses, and the direct kernel with its weights broadcast from
    shared memory or by warp shuffles (forced with acnn_conv2d_force_path)."""
    import torch
    from activation_cnn_gb300 import acnn as A
    from activation_cnn_gb300 import inputs as G
    out = {}
    for name, (n, c, h, w, co, layout, dt, act) in {
            "rgb_stem_8x640x640_3to32_s2_bf16_nhwc": (8, 3, 640, 640, 32, G.NHWC, G.BF16, A.ACT_RELU),
            "frame_input_7x272x480_7to120_s2_f16_nchw": (1, 7, 272, 480, 120, G.NCHW, G.F16,
                                                        A.ACT_PRELU)}.items():
        x = G.tensor(91, name, G.activation_shape(layout, n, c, h, w), "uniform", 0.0, 1.0,
                     dtype=dt).to(dev)
        wt = G.conv_weight(91, name, co, c, 3, 3, layout, dt).to(dev)
        b = G.conv_bias(91, name, co).to(dev)
        al = G.prelu_alpha(91, name, co).to(dev)
        d = A.conv_desc(x, co, 3, 3, 2, 1, layout)
        y = torch.empty(A.conv_out_shape(d), dtype=x.dtype, device=dev)
        flops = 2.0 * y.numel() * c * 9  # y elements x (c_in x 3 x 3) multiply-adds
        res = {}
        for label, (path, variant) in {"packed_tensor_core": (0, 0), "direct_smem_weights": (4, 0),
                                       "direct_shfl_weights": (4, 1)}.items():
            A.acnn_conv2d_force_path(path, variant)
            ws_bytes = A.acnn_conv2d_workspace_size(d)
            ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

            def fn(s, ws=ws, ws_bytes=ws_bytes):
                A.check(A.acnn_conv2d_fused(d, x, wt, b, al, None, A.RES_NONE, act, y, ws,
                                            ws_bytes, s), name)
            t = time_call(fn, stream, flush, reps)
            res[label] = {"path": A.acnn_conv2d_path(d), "us": round(t * 1e6, 2),
                          "TFLOP_s": round(flops / t / 1e12, 2)}
        A.acnn_conv2d_force_path(0, 0)
        out[name] = res
    return out


def measure_config(name, dev, stream, flush, steps, pk):
    """One of the other workloads (single conv, fp32 stem, bottleneck blocks,
    frame stack), timed like the main one: step time, then every op's share of
    it against its own roof."""
    import torch
    from activation_cnn_gb300 import acnn as A
    net = build_net(name, dev)
    with torch.cuda.stream(stream):
        net.run_eager(stream)
    stream.synchronize()
    st = A.acnn_last_device_status(stream.cuda_stream)
    if st != 0:
        raise RuntimeError(f"{name}: device status after eager pass: {A.status_string(st)}")
    net.capture(stream)
    for _ in range(3):
        net.replay(stream)
    step = statistics.mean(time_steps(net, stream, steps, flush))
    rows = apportion(time_ops(net, stream, max(3, min(steps, 20)), flush),
                     time_sections(net, stream, max(3, min(steps, 20)), flush), step)
    net.release()
    st = A.acnn_last_device_status(stream.cuda_stream)
    if st != 0:
        raise RuntimeError(f"{name}: device status after timing: {A.status_string(st)}")
    out = {"workload": name, "us_per_step": round(step * 1e6, 2),
           "steps": steps, "dtype": dtype_name(net),
           "layout": "NHWC" if net.layout == 0 else "NCHW", "batch": net.batch}
    unit = "frames/s" if name.startswith("frame") else "img/s"
    out[unit.replace("/", "_")] = round(net.batch / step, 2)
    conv = [r for r in rows if r["kind"] == "conv"]
    if conv:
        ct = sum(r["t"] for r in conv)
        out["conv_TFLOP_s"] = round(sum(r["flops"] for r in conv) / ct / 1e12, 3)
    out["ops"] = [op_summary(r, pk) for r in rows]
    del net
    torch.cuda.empty_cache()
    return out


def end_to_end(net, stream, steps, world):
    """The workload fed from pinned host memory and read back to it, every step.

    Step i's input is copied host -> device on a copy stream into one of two
    device staging buffers while step i-1 computes; the compute stream copies
    it into the network's input (device to device) and replays the graphs; the
    step's output maps go to a device staging buffer and then device -> host
    on a second copy stream while step i+1 computes.  The timed region runs
    from the first host -> device copy to the end of the last device -> host
    copy.  No L2 flush between steps: each step moves ~2.7 GB through DRAM,
    far more than the 129 MB L2.  A workload whose step moves less than 4x the
    L2 is measured step by step instead, with an L2 flush before each step
    outside the timed interval (end_to_end_serial)."""
    import torch
    from activation_cnn_gb300 import replicas as R
    in_names = list(net.inputs)
    outs = net.output_tensors()
    host_in = {k: net.inputs[k].detach().cpu().pin_memory() for k in in_names}
    host_out = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
                for _ in range(2)]
    in_stage = [{k: torch.empty_like(net.inputs[k]) for k in in_names} for _ in range(2)]
    out_stage = [[torch.empty_like(o) for o in outs] for _ in range(2)]
    ev = lambda: torch.cuda.Event()
    h2d_done, in_free, step_done, d2h_done = ([ev(), ev()] for _ in range(4))
    cs = torch.cuda.Stream(device=stream.device)  # host -> device
    ds = torch.cuda.Stream(device=stream.device)  # device -> host

    def run(k_steps):
        for i in range(k_steps):
            b = i % 2
            cs.wait_event(in_free[b])  # step i-2 has taken its input out of slot b
            with torch.cuda.stream(cs):
                for k in in_names:
                    in_stage[b][k].copy_(host_in[k], non_blocking=True)
            h2d_done[b].record(cs)
            stream.wait_event(h2d_done[b])
            with torch.cuda.stream(stream):
                for k in in_names:
                    net.inputs[k].copy_(in_stage[b][k], non_blocking=True)
                in_free[b].record(stream)
                net.replay(stream)
                stream.wait_event(d2h_done[b])  # step i-2's maps have left slot b
                for o, st in zip(outs, out_stage[b]):
                    st.copy_(o, non_blocking=True)
            step_done[b].record(stream)
            ds.wait_event(step_done[b])
            with torch.cuda.stream(ds):
                for st, h in zip(out_stage[b], host_out[b]):
                    h.copy_(st, non_blocking=True)
            d2h_done[b].record(ds)

    if sum(op.bytes for op in net.ops) < 4 * L2_BYTES:
        return end_to_end_serial(net, stream, steps, world, host_in, host_out[0])
    run(3)  # warm-up
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cs)
    run(steps)
    e1.record(ds)
    torch.cuda.synchronize()
    tot = R.max_over_ranks(e0.elapsed_time(e1) * 1e-3)
    bi = sum(t.numel() * t.element_size() for t in host_in.values())
    bo = sum(t.numel() * t.element_size() for t in host_out[0])
    return {"value": round(net.batch * world * steps / tot, 3), "unit": "img/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "pipelined": "host copies of steps i-1/i+1 overlap step i (two copy streams)",
            "l2": "not flushed: a step's algorithmic traffic exceeds 4x the 129 MB L2"}


def end_to_end_serial(net, stream, steps, world, host_in, host_out):
    """One step at a time: flush L2, then (timed) host -> device input, the
    graphs, device -> host output maps, all on the launching stream."""
    import torch
    from activation_cnn_gb300 import replicas as R
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=stream.device)
    outs = net.output_tensors()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tot = 0.0
    for _ in range(steps):
        with torch.cuda.stream(stream):
            flush_buf.add_(1)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for k, h in host_in.items():
                net.inputs[k].copy_(h, non_blocking=True)
            net.replay(stream)
            for o, h in zip(outs, host_out):
                h.copy_(o, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
        tot += e0.elapsed_time(e1) * 1e-3
    tot = R.max_over_ranks(tot)
    bi = sum(t.numel() * t.element_size() for t in host_in.values())
    bo = sum(t.numel() * t.element_size() for t in host_out)
    return {"value": round(net.batch * world * steps / tot, 3), "unit": "img/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "pipelined": False,
            "l2": "flushed before each step, outside the timed interval"}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from activation_cnn_gb300 import acnn as A
    from activation_cnn_gb300 import build as B
    from activation_cnn_gb300 import replicas as R

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    B.build()
    A.lib()
    net = build_net(args.workload, dev, args.batch)
    stream = torch.cuda.Stream(device=dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush():
        # read + write of a buffer 4x the L2, enqueued on the launching stream so
        # it completes after the previous step and before the next start event
        # (a flush on another stream would overlap the previous step's tail)
        with torch.cuda.stream(stream):
            flush_buf.add_(1)

    # one eager pass (checks every call), then one CUDA graph per section
    with torch.cuda.stream(stream):
        net.run_eager(stream)
    stream.synchronize()
    st = A.acnn_last_device_status(stream.cuda_stream)
    if st != 0:
        raise RuntimeError(f"device status after eager pass: {A.status_string(st)}")
    net.capture(stream)
    for _ in range(max(args.warmup, 3)):
        net.replay(stream)
    stream.synchronize()

    # ------------------------------------------------ timed region (device time)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    R.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush()
        starts[i].record(stream)
        net.replay(stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    R.barrier()
    step_s = [a.elapsed_time(b) * 1e-3 for a, b in zip(starts, ends)]
    total = sum(step_s)
    total = R.max_over_ranks(total)
    st = A.acnn_last_device_status(stream.cuda_stream)
    if st != 0:
        raise RuntimeError(f"device status after timed region: {A.status_string(st)}")

    imgs = net.batch * world * args.steps
    value = imgs / total
    ms_per_step = 1e3 * total / args.steps
    conv_tflops = net.conv_flops() * world * args.steps / total / 1e12

    # ------------------------------------------------ roofline of the dominant kernel
    # Per-op times apportioned from the step itself (apportion): the sections
    # replayed alone give each section's share of the step, the event-bracketed
    # per-op times each op's share of its section.
    pk = peaks()
    nrep = max(3, min(args.steps, 10))
    sec_t = time_sections(net, stream, nrep, flush)
    rows = apportion(time_ops(net, stream, nrep, flush), sec_t, total / args.steps)
    # each section's share of the measured step (sections replayed alone after
    # an L2 flush give the shares)
    sec_tot = sum(sec_t.values())
    sections_us = {k: round(1e6 * (total / args.steps) * v / sec_tot, 1) for k, v in sec_t.items()}
    ig = [r for r in rows if r["kind"] == "conv" and r["path"] in (1, 2)]
    ig_flops = sum(r["flops"] for r in ig)
    ig_t = sum(r["t"] for r in ig)
    achieved = ig_flops / ig_t / 1e12 if ig_t > 0 else 0.0
    peak = pk["bf16_burst"]
    step_s = total / args.steps
    roofline = {"kernel": "igemm_conv_kernel (tcgen05 implicit-GEMM conv)",
                "bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4) if peak else None,
                "peak_source": f"{pk['source']} bf16 burst (a step lasts "
                               f"{1e3 * step_s:.2f} ms)",
                "frac_of_sustained": round(achieved / pk["bf16_sustained"], 4),
                "traffic": conv_traffic(args.workload, args.batch),
                "traffic_how": CONV_TRAFFIC["how"],
                "algorithmic_bytes_per_launch": round(sum(r["bytes"] for r in ig) / max(1, len(ig))),
                "launches_per_step": len(ig),
                "flops_per_launch": ig_flops / max(1, len(ig)),
                "avg_launch_us": round(1e6 * ig_t / max(1, len(ig)), 3),
                "kernel_us_per_step": round(1e6 * ig_t, 1),
                "step_us": round(1e6 * step_s, 1),
                "share_of_step": round(ig_t / step_s, 4),
                "time_source": "CUDA events on the launching stream: the timed steps, each "
                               "section graph replayed alone, and each op bracketed by event "
                               "nodes; the step is split over the ops by section share x "
                               "op share of its section"}
    # each conv launch against its own roof, max(FLOPs / tensor peak, bytes /
    # HBM peak): the fraction of the attainable time the launches achieve
    ideal = sum(max(r["flops"] / (peak * 1e12), r["bytes"] / (pk["hbm"] * 1e9)) for r in ig)
    roofline["attainable"] = {"ideal_us_per_step": round(ideal * 1e6, 1),
                              "measured_us_per_step": round(ig_t * 1e6, 1),
                              "frac": round(ideal / ig_t, 4) if ig_t > 0 else None,
                              "per_launch_roof": "max(flops / tensor peak, bytes / hbm peak)"}

    # ------------------------------------------------ end to end through host buffers
    e2e = None
    if args.e2e:
        e2e = end_to_end(net, stream, args.steps, world)
    net.release()

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "img/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype_name(net),
        "data": "synthetic (seeded; He-normal weights, BN folded into bias)",
        "config": workload_config(args.workload, net, world),
        "conv_tflops": round(conv_tflops, 2),
        "conv_frac_bf16_peak": round(conv_tflops / pk["bf16_burst"], 4),
        "conv_gflop_per_step": round(net.conv_flops() / 1e9, 2),
        "roofline": roofline, "e2e": e2e, "sections_us": sections_us,
        "gpu_launches": launches_per_step(net) * args.steps,
        "clocks": clk, "wall_s_timed": round(t_wall, 3),
    }
    # memory-bound companions: algorithmic bytes / apportioned time vs HBM
    mem = {}
    for r in rows:
        if r["kind"] in ("pool", "resize", "concat", "prep", "deconv"):
            k = mem.setdefault(r["kind"], {"launches": 0, "bytes": 0.0, "t": 0.0})
            k["launches"] += 1
            k["bytes"] += r["bytes"]
            k["t"] += r["t"]
    line["memops"] = {k: {"launches": v["launches"], "GB_s": round(v["bytes"] / v["t"] / 1e9, 1),
                          "frac_hbm": round(v["bytes"] / v["t"] / 1e9 / pk["hbm"], 4),
                          "us_per_step": round(1e6 * v["t"], 1)}
                      for k, v in mem.items()}
    line["memops_peak"] = f"{pk['source']} HBM copy {pk['hbm']} GB/s"
    direct = [r for r in rows if r["kind"] == "conv" and r["path"] == 0]
    if direct:
        ds = sum(r["t"] for r in direct)
        line["direct_conv"] = {"launches": len(direct), "us_per_step": round(1e6 * ds, 1),
                               "TFLOP_s": round(sum(r["flops"] for r in direct) / ds / 1e12, 2)}
    if args.layers:
        line["layers"] = [op_summary(r, pk) for r in rows]
    # the other workloads, each timed the same way
    if args.configs and args.workload == "backbone" and args.batch in (None, 8):
        line["configs"] = {name: measure_config(name, dev, stream, flush, 50, pk)
                           for name in ("conv1", "stem", "block", "block_down", "frame")}
        line["tiny_cin_conv"] = tiny_cin_compare(dev, stream, flush)
    return line


def dtype_name(net):
    from activation_cnn_gb300 import inputs as G
    return {G.F32: "f32", G.F16: "f16", G.BF16: "bf16"}[net.dtype]


# ---------------------------------------------------------------- oracle arms
def oracle_sample(workload, kind):
    """(callable, fraction of one step's images it covers, description)."""
    import torch
    from activation_cnn_gb300 import inputs as G
    from oracle import models as M
    from oracle import oracle as O
    O.build()
    if workload != "backbone":
        raise SystemExit("the oracle baseline is implemented for the backbone workload")
    # cpu_baseline: three full 640x640 images (3/8 of a step, ~10 s on 16 cores);
    # reference steps: one 160x160 image, i.e. 1/16 of one image's conv work (every
    # op scales with the pixel count)
    side, n = (640, 3) if kind == "baseline" else (160, 1)
    x = G.tensor(1238, "x", (n, side, side, 3), "uniform", 0.0, 1.0, dtype=G.BF16)
    x64 = x.to(torch.float64).numpy()
    frac = n * (side * side) / (640 * 640)
    desc = (f"oracle backbone+neck forward (fp64, bf16 storage emulation) on {n} "
            f"{side}x{side}x3 image(s) = {frac:g} of one image's work, {O.nthreads()} threads")
    return (lambda: M.backbone(x64)), frac, desc


def cpu_baseline(workload):
    from oracle import oracle as O
    fn, frac, desc = oracle_sample(workload, "baseline")
    t0 = time.perf_counter()
    fn()
    dt = time.perf_counter() - t0
    return {"value": round(frac / dt, 5), "unit": "img/s", "cores": O.nthreads(),
            "kind": "oracle", "sample": desc, "seconds": round(dt, 2)}


def run_reference(args):
    from oracle import oracle as O
    fn, frac, desc = oracle_sample(args.workload, "reference")
    for _ in range(args.warmup):
        fn()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn()
    dt = time.perf_counter() - t0
    value = frac * args.steps / dt
    return {"metric": METRIC, "value": round(value, 5), "unit": "img/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * dt / args.steps, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": args.workload, "image": "640x640x3",
                       "sample_per_step": desc},
            "cpu_baseline": {"value": round(value, 5), "unit": "img/s", "cores": O.nthreads(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 5), "unit": "img/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="backbone",
                    choices=["backbone", "backbone_csp", "block", "block_down", "stem", "conv1", "frame",
                             "frame_out", "frame_tfact"])
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--layers", action="store_true", help="add per-op timings")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the other workloads' sub-objects (single conv, fp32 stem, "
                         "bottleneck blocks, frame stack)")
    ap.add_argument("--batch", type=int, default=None,
                    help="batch per GPU of the backbone (default 8) or a bottleneck block (default 4); "
                         "other sizes for profiler captures")
    args = ap.parse_args()

    from activation_cnn_gb300 import replicas as R
    rank, world, local_rank = R.env()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if args.cpu_baseline and args.workload == "backbone":
            line["cpu_baseline"] = cpu_baseline(args.workload)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
