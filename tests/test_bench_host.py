"""Host logic of bench.py that decides what a bench line reports (no GPU).

* the DRAM traffic of a kernel is taken from profiles/traffic.json only while
  the recorded source hash matches the kernel's current sources;
* the clock summary turns NVML clock-event reason bits and nvidia-smi CSV
  rows into the reason names the timing rules name.
"""
import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_traffic_record_follows_the_source_hash(bench):
    import json
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for kernel in ("spec_verify", "commit_kernel"):
        assert kernel in rec
        h = rec[kernel]["source_hash"]
        # the sources the counters were taken on give the recorded bytes ...
        assert bench.traffic_record(kernel, h) == float(rec[kernel]["dram_bytes_per_launch"])
        # ... any other source gives no traffic figure
        assert bench.traffic_record(kernel, "0" * 16) is None
    assert bench.traffic_record("no_such_kernel", "0" * 16) is None


def test_kernel_source_hash_changes_with_the_text(bench, tmp_path, monkeypatch):
    csrc = tmp_path / "speculative_decoding_verify_07_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cu").write_text("int x;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h1 = bench.kernel_source_hash(["a.cu"])
    (csrc / "a.cu").write_text("int y;\n")
    h2 = bench.kernel_source_hash(["a.cu"])
    assert len(h1) == 16 and h1 != h2


def test_clock_summary_from_nvml_samples(bench):
    c = bench.ClockSampler(0)
    c.thread = object()   # as if the NVML thread had run
    # (sm MHz, max MHz, reason bits): power cap (kept, noted), then hardware
    # and software thermal slowdowns (a rejected run)
    c.samples = [(2070.0, 2070.0, 0x0), (2055.0, 2070.0, 0x4), (1980.0, 2070.0, 0x8 | 0x20 | 0x40)]
    s = c.summary()
    assert s["sm_mhz"] == 2055.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert s["source"] == "nvml"
    c.samples = [(2070.0, 2070.0, 0x1)]   # idle bit alone is no reason
    assert c.summary()["reasons"] == []


def test_clock_summary_from_nvidia_smi_rows(bench, tmp_path):
    c = bench.ClockSampler(0)
    c.path = str(tmp_path / "clocks.csv")
    c.proc = object()   # as if nvidia-smi had written the file
    (tmp_path / "clocks.csv").write_text(
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"
        "0, 2062, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active\n"
        "garbage line\n"
        "0, 1800, 2070, 1400.0, 0x8, Active, Not Active, Not Active, Active\n")
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2062.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert s["source"] == "nvidia-smi"
