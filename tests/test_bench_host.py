"""Host-side logic of bench.py that needs no GPU: the clock-sample summary
that decides whether a timed run is kept, the launch count per step and the
traffic record's source-hash check."""
from __future__ import annotations

import importlib
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
bench = importlib.import_module("bench")


def _line(t: float, mhz: int, reasons=("Not Active",) * 4) -> str:
    whole = int(t)
    stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(whole)) + ".%03d" % int((t - whole) * 1000)
    return ", ".join([stamp, "0", str(mhz), "2070", "950.00", "0x0000000000000000", *reasons])


def test_clock_summary_takes_the_timed_region_only():
    t0 = float(int(time.time()))
    lines = [_line(t0 - 5, 900), _line(t0 + 0.5, 2070), _line(t0 + 1.0, 2040), _line(t0 + 1.5, 2070),
             _line(t0 + 9, 900), "garbage line", ""]
    rows = bench.parse_clock_lines(lines)
    assert len(rows) == 5
    s = bench.summarize_clocks(rows, t0 + 0.4, t0 + 1.6)
    assert s["samples_inside_timed_region"] == 3 and s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == []


def test_clock_summary_reports_throttle_reasons():
    t0 = float(int(time.time()))
    hot = ("Active", "Not Active", "Active", "Not Active")  # hw_slowdown, sw_thermal_slowdown
    rows = bench.parse_clock_lines([_line(t0 + 0.5, 1500, hot), _line(t0 + 0.6, 1600)])
    s = bench.summarize_clocks(rows, t0, t0 + 1)
    assert s["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples_is_none_and_nearest_samples_otherwise():
    assert bench.summarize_clocks([], 0.0, 1.0) is None
    t0 = float(int(time.time()))
    rows = bench.parse_clock_lines([_line(t0 - 3, 2070), _line(t0 + 30, 2000)])
    s = bench.summarize_clocks(rows, t0, t0 + 0.01)
    assert s["samples_inside_timed_region"] == 0 and s["samples"] == 2


def test_launches_per_step():
    assert bench.launches_per_step(1) == 3 and bench.launches_per_step(64) == 3
    assert bench.launches_per_step(65) == 9


def test_traffic_record_requires_matching_sources(tmp_path, monkeypatch):
    path = os.path.join(ROOT, "profiles", "traffic.json")
    rec = json.load(open(path))
    # the committed record carries the hash of the library sources it was taken on
    assert all(len(v["csrc_sha256"]) == 64 for v in rec.values())
    fake_root = tmp_path
    (fake_root / "profiles").mkdir()
    bad = {k: dict(v, csrc_sha256="0" * 64) for k, v in rec.items()}
    (fake_root / "profiles" / "traffic.json").write_text(json.dumps(bad))
    monkeypatch.setattr(bench, "ROOT", str(fake_root))
    assert bench.traffic_record("decode1") is None
