"""bench.py's host-side helpers on CPU: the clock summary taken from nvidia-smi samples.

The summary decides the `clocks` object of the benchmark line (median SM clock under load,
maximum clock, throttle reasons seen), so its parsing is checked here on synthetic lines in
nvidia-smi's `--format=csv,noheader,nounits` layout, without a GPU.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(sm, smax=2070, power=900.0, active="0x0000000000000000", hw="Not Active",
          hw_thermal="Not Active", sw_thermal="Not Active", sw_power="Not Active"):
    return f"0, {sm}, {smax}, {power}, {active}, {hw}, {hw_thermal}, {sw_thermal}, {sw_power}"


def _summary(lines):
    s = bench.ClockSampler("0")
    s.lines = list(lines)
    return s.summary()


def test_loaded_median_and_no_reasons():
    out = _summary([_line(2070), _line(2070), _line(2055), _line(2070)])
    assert out == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 4}


def test_idle_samples_left_out_of_the_median():
    # samples before the load starts (idle clocks) do not pull the median down
    out = _summary([_line(345), _line(345), _line(2070), _line(2070), _line(2070)])
    assert out["sm_mhz"] == 2070.0
    assert out["samples"] == 5


def test_throttle_reasons_are_reported():
    out = _summary([_line(1980, sw_power="Active"), _line(2070),
                    _line(1800, hw_thermal="Active"), _line(2000, hw="Active")])
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]
    out = _summary([_line(2070, sw_thermal="Active")])
    assert out["reasons"] == ["sw_thermal_slowdown"]


def test_no_samples_and_unparsable_samples():
    assert _summary([])["reasons"] == ["nvidia-smi unavailable"]
    bad = _summary(["[N/A], [N/A]", "0, [Not Supported], 2070, 1, 0x0, x, x, x, x"])
    assert bad["reasons"] == ["no parsable samples"] and bad["samples"] == 0


def test_aggregate_is_whole_job_throughput():
    # units all ranks processed over the slowest rank's time
    assert bench.aggregate(100.0, 2.0, 1) == 50.0
    assert bench.aggregate(100.0, 2.0, 4) == 200.0


def test_profiled_fields_follow_the_kernel_sources(monkeypatch):
    # traffic and achieved occupancy come from captures of the kernels as they are now; once
    # a kernel source changes they must read as unmeasured (None), not as stale numbers
    name = "cconv_bwd_ls_kernel<4, 12, 4, 8, 1, 0>"
    upd = "cconv_update_kernel<8, 4, 3, 4, 0, 256>"
    current = {fam: bench.sources_sha16(files) for fam, files in bench.OCCUPANCY_SOURCES.items()}
    monkeypatch.setitem(bench.BWD_TRAFFIC, "sources_sha16", bench.sources_sha16())
    monkeypatch.setitem(bench.ACHIEVED_OCCUPANCY, "sources_sha16", dict(current))
    assert bench.bwd_traffic() == bench.BWD_TRAFFIC["bytes_per_call"]
    assert bench.achieved_occupancy(name) == bench.ACHIEVED_OCCUPANCY["pct"][name]
    assert bench.achieved_occupancy(upd) == bench.ACHIEVED_OCCUPANCY["pct"][upd]
    assert bench.achieved_occupancy("cconv_bwd_reduce1_kernel") is None  # not captured
    assert bench.achieved_occupancy("some_other_kernel") is None
    monkeypatch.setitem(bench.BWD_TRAFFIC, "sources_sha16", "0" * 16)
    assert bench.bwd_traffic() is None
    # a change in one family's sources voids that family's figures only
    monkeypatch.setitem(bench.ACHIEVED_OCCUPANCY, "sources_sha16", dict(current, update="0" * 16))
    assert bench.achieved_occupancy(upd) is None
    assert bench.achieved_occupancy(name) == bench.ACHIEVED_OCCUPANCY["pct"][name]
    monkeypatch.setitem(bench.ACHIEVED_OCCUPANCY, "sources_sha16", dict(current, bwd="0" * 16))
    assert bench.achieved_occupancy(name) is None
    assert bench.achieved_occupancy(upd) == bench.ACHIEVED_OCCUPANCY["pct"][upd]
