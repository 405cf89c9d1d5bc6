"""Host-side pieces of the benchmark that need no GPU: the DRAM-traffic figure
is reported only while the kernel sources it was measured on are unchanged,
the algorithmic byte counts follow the per-element figures, and the clock
summary keeps only loaded samples and the throttle reasons seen."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_is_null_once_a_source_changed(monkeypatch):
    entry = dict(bench.TRAFFIC["fp8_to_mx"])
    monkeypatch.setitem(bench.TRAFFIC, "fp8_to_mx", dict(entry, src_sha=bench._src_hash(entry["src"])))
    assert bench._traffic("fp8_to_mx") == entry["bytes_per_launch"]
    monkeypatch.setitem(bench.TRAFFIC, "fp8_to_mx", dict(entry, src_sha="0" * 16))
    assert bench._traffic("fp8_to_mx") is None
    assert bench._traffic("no_such_kernel") is None


def test_algorithmic_bytes_per_element():
    n = bench.ROWS * bench.COLS
    # 1 + 4/128 in, 0.5 + 1/32 out  (and the reverse for the conversion back)
    assert bench.bytes_fp8_to_mx(bench.ROWS, bench.COLS) == n * 1.5625
    assert bench.bytes_mx_to_fp8(bench.ROWS, bench.COLS) == n * 1.5625


def test_clock_summary_keeps_loaded_samples_and_reasons(monkeypatch):
    class FakeProc:
        def __init__(self, text):
            self.text = text

        def terminate(self):
            pass

        def communicate(self, timeout=None):
            return self.text, ""

    lines = ["0, 2070, 2070, 900, 0x0, Not Active, Not Active, Not Active, Active",
             "0, 2070, 2070, 950, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 345, 2070, 100, 0x0, Not Active, Not Active, Not Active, Not Active",   # idle: dropped
             "garbage line"]
    c = bench.ClockSampler(0)
    c.proc = FakeProc("\n".join(lines))
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    out = c.stop()
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070 and out["samples"] == 2
    assert out["reasons"] == ["sw_power_cap"]
