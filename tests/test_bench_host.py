"""Host-side logic of bench.py (no GPU): the committed DRAM-traffic record is reported only
for the kernel source and options it was captured with; the clock sampler's parsing."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_record_matches_only_its_capture(monkeypatch):
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    key = "gemm_n256_c1_clc_square"
    rg = rec["kernels"][key]["raster_group"]
    other = 8 if rg != 8 else 16
    monkeypatch.setattr(bench, "kernel_hash", lambda: rec["kernel_hash"])
    assert bench.traffic_for(key, rg, 0) == float(rec["kernels"][key]["dram_bytes_per_launch"])
    assert bench.traffic_for(key, other, 0) is None       # other raster band
    assert bench.traffic_for(key, rg, 4) is None          # other prefetch distance
    assert bench.traffic_for("no_such_kernel", rg, 0) is None
    monkeypatch.setattr(bench, "kernel_hash", lambda: "0" * 16)
    assert bench.traffic_for(key, rg, 0) is None          # kernel changed since the capture


def test_clock_sampler_parses_nvidia_smi_lines():
    s = bench.ClockSampler.__new__(bench.ClockSampler)

    class P:
        def terminate(self):
            pass

        def communicate(self, timeout=None):
            return ("0, 1800, 2070, 1300.5, 0x4, Not Active, Not Active, Not Active, Active\n"
                    "0, 1900, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, Active\n"
                    "0, 2000, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active\n", "")

    s.proc = P()
    out = s.stop()
    assert out["sm_mhz"] == 1900 and out["sm_max_mhz"] == 2070 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]
