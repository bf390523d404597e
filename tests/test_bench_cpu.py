"""Host-side pieces of bench.py: the traffic record, launch counting, clock parsing."""
import os
import tempfile

import pytest

import bench


def test_traffic_only_for_the_kernel_source_it_was_taken_on(monkeypatch):
    """bench reports the conv kernel's per-launch DRAM bytes only for the
    default backbone step and only while the kernel source hash matches the one
    the counters were taken on."""
    monkeypatch.setattr(bench, "CONV_TRAFFIC",
                        {"kernel_sha16": bench.kernel_source_hash(), "bytes_per_launch": 4.2e7,
                         "how": "test"})
    assert bench.conv_traffic("backbone", None) == 4.2e7
    assert bench.conv_traffic("backbone", 2) is None
    assert bench.conv_traffic("block", None) is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.conv_traffic("backbone", None) is None


def test_apportion_splits_the_step_over_ops():
    """Section shares x op shares: the ops' times sum to the step, every op
    keeps its share of its own section, and an op's time never exceeds the
    step (so a roofline fraction computed from it follows from the step)."""
    rows = [{"section": "a", "s": 3.0}, {"section": "a", "s": 1.0},
            {"section": "b", "s": 2.0}]
    out = bench.apportion(rows, {"a": 6.0, "b": 2.0}, 4.0)
    ts = [r["t"] for r in out]
    assert abs(sum(ts) - 4.0) < 1e-12
    assert abs(ts[0] - 4.0 * 0.75 * 0.75) < 1e-12 and abs(ts[1] - 4.0 * 0.75 * 0.25) < 1e-12
    assert abs(ts[2] - 1.0) < 1e-12
    assert max(ts) <= 4.0


def test_op_summary_fractions():
    pk = {"bf16_burst": 2000.0, "bf16_sustained": 1700.0, "hbm": 7000.0}
    conv = {"name": "c", "kind": "conv", "path": 1, "flops": 2e12 * 1e-3, "bytes": 1e6,
            "t": 2e-6}
    d = bench.op_summary(conv, pk)
    assert d["TFLOP_s"] == 1000.0 and d["frac_tensor_peak"] == 0.5
    # roof = max(2e9 / 2e15, 1e6 / 7e12) = 1 us of 2 us
    assert abs(d["attainable_frac"] - 0.5) < 1e-4
    pool = {"name": "p", "kind": "pool", "path": None, "flops": 0.0, "bytes": 7e6, "t": 2e-6}
    d = bench.op_summary(pool, pk)
    assert d["GB_s"] == 3500.0 and d["frac_hbm"] == 0.5
    direct = {"name": "d", "kind": "conv", "path": 0, "flops": 1e8, "bytes": 1e6, "t": 1e-5}
    assert abs(bench.op_summary(direct, pk)["frac_fp32_ffma"] -
               1e8 / 1e-5 / 1e12 / bench.FP32_FFMA_TFLOPS) < 1e-4


class _Op:
    def __init__(self, launches):
        self.launches = launches


class _Net:
    def __init__(self, counts):
        self.ops = [_Op(c) for c in counts]


def test_launches_per_step_sums_each_ops_count():
    assert bench.launches_per_step(_Net([1, 2, 1, 1])) == 5
    assert bench.launches_per_step(_Net([])) == 0


class _Proc:
    def terminate(self):
        pass

    def wait(self):
        return 0


def _sampler_with(lines):
    s = bench.ClockSampler(0)
    fd, s.path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.proc = _Proc()
    return s


def test_clock_samples_median_and_reasons(monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda _: None)
    s = _sampler_with([
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ])
    path = s.path
    r = s.stop()
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["samples"] == 3
    assert r["reasons"] == ["sw_power_cap"]
    assert not os.path.exists(path)


def test_clock_samples_flag_thermal_slowdown(monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda _: None)
    s = _sampler_with(["0, 1500, 2070, 1000.0, 0x40, Active, Active, Not Active, Not Active"])
    r = s.stop()
    assert r["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_clock_sampler_without_nvidia_smi():
    s = bench.ClockSampler(0)
    s.proc = None
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


@pytest.mark.parametrize("wl", ["backbone", "frame_out", "frame_tfact", "backbone_csp"])
def test_workloads_are_bench_choices(wl):
    from activation_cnn_gb300 import network as N
    assert wl in N.WORKLOADS
