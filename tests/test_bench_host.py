"""Host logic of the benchmark that needs no GPU: the clock/throttle record
parsed from nvidia-smi lines, and the ncu traffic figure taken from a profile
summary only for the kernel source it was captured on."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_clocks_median_max_and_active_reasons():
    lines = "\n".join([
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 2040, 2070, 1100.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1995, 2070, 1390.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ])
    c = bench.parse_clocks(lines)
    assert c["samples"] == 3
    assert c["sm_mhz"] == 2040.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]


def test_clocks_thermal_reasons_are_reported():
    lines = "0, 1500, 2070, 1400, 0x68, Active, Active, Active, Not Active"
    c = bench.parse_clocks(lines)
    assert c["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clocks_no_samples():
    assert bench.parse_clocks("") == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                                      "samples": 0}


def test_profile_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k.md").write_text("kernel source sha256[:16]: 0123456789abcdef\n"
                               "dram bytes per launch (full workload): 9.229e9\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("k.md", "0123456789abcdef") == 9.229e9
    assert bench.profile_traffic("k.md", "fedcba9876543210") is None
    assert bench.profile_traffic("missing.md", "0123456789abcdef") is None



def test_profile_traffic_per_call_labels(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "p.md").write_text("kernel source sha256[:16]: 0123456789abcdef\n"
                               "dram bytes per call (qkvg, decode_b64_h32_x256): 238811392\n"
                               "dram bytes per call (o, decode_b64_h32_x256): 62164992\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = "0123456789abcdef"
    assert bench.profile_traffic("p.md", sha, "per call (qkvg, decode_b64_h32_x256)") == 238811392.0
    assert bench.profile_traffic("p.md", sha, "per call (o, decode_b64_h32_x256)") == 62164992.0
    assert bench.profile_traffic("p.md", sha, "per call (o, prefill_b8_h64_t8192)") is None
    assert bench.profile_traffic("p.md", sha) is None   # no per-launch line in this file
