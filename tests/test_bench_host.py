"""Host-side pieces of bench.py that need no GPU: the profiled DRAM traffic is
reported only while it was taken on the current kernel source, and the clock
summary flags every throttle reason it was given."""
import os
import shutil

import bench


def test_traffic_is_dropped_once_the_kernel_source_changes(tmp_path, monkeypatch):
    src = tmp_path / "paged_decode.cu"
    shutil.copy(bench.DECODE_SRC, src)
    summary = tmp_path / "traffic.txt"
    summary.write_text("# a summary taken on this source\n"
                       f"source_sha256_16: {bench.source_digest(str(src))}\n"
                       "dram_bytes_per_launch: 3229509120\n")
    monkeypatch.setattr(bench, "DECODE_SRC", str(src))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(summary))
    assert bench.profiled_traffic() == 3229509120.0
    with open(src, "a") as f:
        f.write("\n// edited\n")
    assert bench.profiled_traffic() is None
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", os.path.join(str(tmp_path), "missing.txt"))
    assert bench.profiled_traffic() is None


def test_clock_summary_reports_throttle_reasons():
    s = bench.ClockSampler(0)
    s.lines = [
        "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1950, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 950.0, 0x0, Not Active, Active, Not Active, Not Active",
        "garbage line",
    ]
    out = s.summary()
    assert out["samples"] == 3 and out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    empty = bench.ClockSampler(0).summary()
    assert empty["reasons"] == ["unsampled"] and empty["samples"] == 0
