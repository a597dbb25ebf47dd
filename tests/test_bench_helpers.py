"""Host-side helpers of bench.py, without a GPU: the clock record taken during the timed region,
the peak lookup, and the rule that DRAM counters count only for the kernel sources they were
taken on."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sampler(first: str, rest: str) -> "bench.ClockSampler":
    cs = bench.ClockSampler(0)
    cs.first, cs.out = first, rest
    return cs


def _row(sm, smax, power, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return f"0, {sm}, {smax}, {power}, 0x0, {hw}, {hwt}, {swt}, {cap}\n"


def test_clock_summary_takes_busy_samples_and_collects_reasons():
    rows = [_row(345, 2070, 90.0)] + [_row(2070, 2070, 900.0)] * 5 + [_row(1980, 2070, 1390.0, cap="Active")]
    s = _sampler(rows[0], "".join(rows[1:])).summary()
    assert s["samples"] == 7
    assert s["sm_max_mhz"] == 2070.0
    assert s["sm_mhz"] == 2070.0                     # the idle 345 MHz sample is not "under load"
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_slowdowns_and_missing_samples():
    s = _sampler("", _row(1200, 2070, 1400.0, hw="Active", swt="Active")).summary()
    assert s["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    s = _sampler("", "").summary()
    assert s["samples"] == 0 and s["reasons"] == ["unsampled"]
    s = _sampler("", "[N/A], [N/A], x, y, z, a, b, c, d\n").summary()   # unparsable rows are skipped
    assert s["samples"] == 0


def test_clock_summary_counts_the_samples_inside_the_timed_region():
    import datetime

    cs = bench.ClockSampler(0)
    cs.t0 = datetime.datetime(2026, 1, 2, 3, 4, 5, 100000)
    cs.t1 = datetime.datetime(2026, 1, 2, 3, 4, 5, 400000)
    before = _row(1500, 2070, 300.0).rstrip("\n") + ", 2026/01/02 03:04:05.050\n"
    inside = [_row(2070, 2070, 900.0).rstrip("\n") + f", 2026/01/02 03:04:05.{ms:03d}\n" for ms in (150, 250, 350)]
    after = _row(1900, 2070, 500.0, cap="Active").rstrip("\n") + ", 2026/01/02 03:04:05.450\n"
    cs.first, cs.out = before, "".join(inside) + after
    s = cs.summary()
    assert s["samples"] == 5 and s["samples_in_region"] == 3
    assert s["sm_mhz"] == 2070.0                       # from the samples inside the region
    assert s["reasons"] == ["sw_power_cap"]             # reasons from every sample


def test_peaks_use_the_measured_file_else_the_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (6800.0, "fallback")
    assert bench.tensor_peak() == (1900.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6790.3, "bf16_tflops": 1890.2}))
    assert bench.peaks() == (6790.3, "measured")
    assert bench.tensor_peak() == (1890.2, "measured")


def test_dram_counters_count_only_for_the_sources_they_were_taken_on(monkeypatch):
    with open(os.path.join(ROOT, "profiles", "decode_kernel_traffic.json")) as f:
        entry = json.load(f)["gqa_batch128"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: entry["source_hash"])
    assert bench.ncu_traffic("gqa_batch128") == {"partition": entry["dram_bytes_per_launch_full"],
                                                  "merge": entry.get("merge_dram_bytes_per_launch")}
    assert bench.ncu_traffic("no_such_workload") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.ncu_traffic("gqa_batch128") is None


def test_source_hash_covers_the_decode_sources():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    for name in bench.DECODE_SOURCES:
        assert os.path.exists(os.path.join(ROOT, "paged_kv_cache_265_gb300", "csrc", name))
