"""Host-side pieces of bench.py: the traffic record, launch counting, clock parsing."""
import os
import tempfile

import pytest

import bench


def test_traffic_record_matches_the_kernel_source():
    """The committed ncu summary carries the conv source's hash; bench reports its
    per-launch DRAM bytes only while the hash matches, and never for a workload
    it was not taken on."""
    assert bench.measured_traffic("no_such_workload") is None
    t = bench.measured_traffic("backbone")
    if t is None:
        pytest.skip("the ncu record was taken on another version of the conv kernel")
    assert 1e6 < t < 1e9


def test_traffic_record_rejects_another_kernel_version(monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.measured_traffic("backbone") is None


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
