"""The benchmark's recorded ncu figures for the draft launch (DRAM traffic and the
warp instruction count of the issue roof): reported only while the engine's
sources hash to the captured version, and the issue roof's arithmetic."""
import json

import bench


def _profile(tmp_path, monkeypatch, traffic_hash, issue_hash):
    (tmp_path / "profiles").mkdir()
    rec = {"dram_bytes_per_launch": 6_500_000_000, "dram_bytes_per_launch_l2_resident": 5_400_000_000,
           "source_hash": traffic_hash,
           "issue": {"source_hash": issue_hash, "warp_instructions": 250_000_000, "logits": 312_500_000}}
    (tmp_path / "profiles" / "draft_engine_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "engine_source_hash", lambda: "current")


def test_figures_of_the_current_sources_are_reported(tmp_path, monkeypatch):
    _profile(tmp_path, monkeypatch, "current", "current")
    assert bench.recorded_engine_traffic() == 6_500_000_000
    assert bench.recorded_engine_traffic(l2_resident=True) == 5_400_000_000
    assert bench.recorded_engine_issue() == 0.8


def test_figures_of_other_sources_are_not(tmp_path, monkeypatch):
    _profile(tmp_path, monkeypatch, "older", "older")
    assert bench.recorded_engine_traffic() is None
    assert bench.recorded_engine_issue() is None
    assert bench.issue_roof(1e9, 1000.0, 2000.0, 100) is None


def test_issue_roof(tmp_path, monkeypatch):
    """0.8 warp instructions a logit, 1e9 logits, 100 SMs of 4 schedulers at 2000 MHz:
    8e8 instructions / (400 x 2000 per us) = 1000 us, half of a 2000 us launch."""
    _profile(tmp_path, monkeypatch, "current", "current")
    roof = bench.issue_roof(1e9, 2000.0, 2000.0, 100)
    assert roof["ideal_us"] == 1000.0 and roof["frac"] == 0.5
    assert bench.issue_roof(1e9, 2000.0, None, 100) is None


def test_no_profile(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_engine_traffic() is None and bench.recorded_engine_issue() is None
