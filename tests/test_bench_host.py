"""Host-side logic of bench.py that decides what the JSON line reports: the
clock summary (samples of the timed region only, throttle reasons) and the
ncu traffic record (reported only while its source hash matches)."""
import importlib.util
import json
import os

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def _row(sm, mx=2070, hw="Not Active", thermal="Not Active", sw_thermal="Not Active",
         power_cap="Not Active"):
    return "0, %d, %d, 900.0, 0x0, %s, %s, %s, %s\n" % (sm, mx, hw, thermal, sw_thermal, power_cap)


def test_clock_summary_keeps_only_the_timed_region():
    b = _bench()
    c = b.ClockSampler(0)
    c.rows = [(0.5, _row(1000, hw="Active")),          # before the timed region
              (1.0, _row(2070)), (1.2, _row(2060)), (1.4, _row(2070, power_cap="Active")),
              (9.0, _row(900, thermal="Active"))]     # after it
    c.t0, c.t1 = 1.0, 1.4
    s = c.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_slowdowns_and_tolerates_bad_rows():
    b = _bench()
    c = b.ClockSampler(0)
    c.rows = [(1.0, _row(1500, hw="Active")), (1.1, "garbage\n"), (1.2, "0, [N/A], 2070, 1, 2, 3, 4, 5, 6\n"),
              (1.3, _row(1600, sw_thermal="Active"))]
    c.t0, c.t1 = 0.0, 2.0
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 1550.0
    assert s["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    empty = b.ClockSampler(0)
    assert empty.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_ncu_traffic_only_for_the_source_it_was_taken_on(tmp_path):
    b = _bench()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(
        {"k:w": {"source_hash": "abc", "dram_bytes_per_launch": 123}}))
    b.ROOT = str(tmp_path)
    assert b.ncu_traffic("k:w", "abc") == 123
    assert b.ncu_traffic("k:w", "abd") is None
    assert b.ncu_traffic("other", "abc") is None
    (tmp_path / "profiles" / "ncu_traffic.json").write_text("not json")
    assert b.ncu_traffic("k:w", "abc") is None


def test_committed_traffic_record_is_well_formed():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    for key, e in d.items():
        assert ":" in key
        assert len(e["source_hash"]) == 16 and int(e["source_hash"], 16) >= 0
        assert isinstance(e["dram_bytes_per_launch"], int) and e["dram_bytes_per_launch"] > 0
        assert os.path.exists(os.path.join(ROOT, e["summary"]))


def test_clock_report_adds_the_load_window_when_the_timed_region_is_short():
    b = _bench()
    c = b.ClockSampler(0)
    c.rows = [(0.5, _row(1000)), (1.01, _row(2070)),
              (2.0, _row(2060)), (2.2, _row(2040, power_cap="Active")), (2.4, _row(2070)),
              (9.0, _row(900, thermal="Active"))]
    c.t0, c.t1 = 1.0, 1.02            # 20 ms timed region: one sample
    r = c.report()
    assert r["samples_timed"] == 1 and r["samples"] == 1 and r["source"] == "timed region"
    c.mark_window(1.9, 2.5)
    r = c.report()
    assert r["samples_timed"] == 1 and r["samples"] == 4
    assert r["sm_mhz"] == 2065.0 and r["reasons"] == ["sw_power_cap"]
    assert "load window" in r["source"]
    c.t0, c.t1 = 1.9, 2.5             # enough samples in the timed region itself
    r = c.report()
    assert r["source"] == "timed region" and r["samples"] == 3
