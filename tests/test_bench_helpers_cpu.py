"""Host helpers of bench.py that the JSON line depends on, checked on CPU.

* The DRAM traffic of a kernel comes from its committed ncu summary only while the kernel's
  sources still hash to the captured ones; otherwise the line must report null.
* The clock summary takes the median SM clock of the samples inside the timed region and
  lists every throttle reason seen active there.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

KERNELS = ("tc_attn_kernel@global_verify", "project_kv_kernel", "accept_kernel", "grouped_conv_kernel",
           "selector_kernel")


def test_every_recorded_traffic_is_current_or_reported_stale():
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert set(KERNELS) <= set(rec)
    for name in KERNELS:
        for f in rec[name]["sources"]:
            assert os.path.exists(os.path.join(ROOT, f)), f
        kernel, _, workload = name.partition("@")
        traffic, note = bench.traffic_from_profiles(kernel, workload or None)
        if rec[name]["source_sha256"] == bench.kernel_source_sha(rec[name]["sources"]):
            assert traffic == rec[name]["dram_bytes_per_launch"] and traffic > 0, name
        else:
            assert traffic is None and "changed" in note, name


def test_traffic_is_null_once_a_source_changes(monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_sha", lambda files: "0" * 64)
    traffic, note = bench.traffic_from_profiles("tc_attn_kernel", "global_verify")
    assert traffic is None and "changed" in note
    # a record of the kernel on another workload never stands for this one
    assert bench.traffic_from_profiles("tc_attn_kernel", "long_draft")[0] is None
    assert bench.traffic_from_profiles("no_such_kernel") == (None, None)


def _line(sm, smax, hw="Not Active", thermal="Not Active", sw_thermal="Not Active", power="Not Active"):
    return f"0, {sm}, {smax}, 900.5, 0x0, {hw}, {thermal}, {sw_thermal}, {power}"


def test_clock_summary_uses_the_timed_region_and_lists_reasons():
    s = bench.ClockSampler(0)
    s.lines = [(1.0, _line(1200, 2070)),                          # before the timed region
               (2.0, _line(2070, 2070)),
               (2.1, _line(2010, 2070, power="Active")),
               (2.2, _line(1980, 2070, hw="Active")),
               (9.0, _line(800, 2070, thermal="Active")),         # after it
               (2.3, "garbled line")]
    out = s.summary(1.5, 3.0)
    assert out["sm_mhz"] == 2010 and out["sm_max_mhz"] == 2070 and out["samples"] == 3
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert out["samples_note"] is None


def test_clock_summary_without_samples_in_the_region():
    s = bench.ClockSampler(0)
    s.lines = [(1.0, _line(2070, 2070))]
    out = s.summary(5.0, 6.0)
    assert out["samples"] == 0 and out["sm_mhz"] == 2070 and out["samples_note"]
    empty = bench.ClockSampler(0).summary(0.0, 1.0)
    assert empty["sm_mhz"] is None and empty["reasons"] == ["no nvidia-smi samples"]


def test_measured_peaks_read_the_driver_file():
    peak, kind = bench.measured_peaks()
    tflops, tkind = bench.measured_tflops()
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        assert (peak, kind) == (float(d["hbm_gbs"]), "measured")
        assert tflops == float(d["bf16_tflops"]) and tkind.startswith("measured")
    else:
        assert kind == "fallback" and tkind == "fallback"
