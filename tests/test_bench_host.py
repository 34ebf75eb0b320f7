"""bench.py's host logic: the committed DRAM-traffic capture is used only while the verify call's
sources are the ones it was taken on, and it scales with the units a launch processes."""

import json

import pytest

import bench


def test_committed_traffic_matches_current_sources():
    with open(bench.PROFILE_TRAFFIC) as f:
        d = json.load(f)
    if d["kernel_src_sha"] != bench.kernel_source_sha():
        pytest.skip("the verify sources changed since the committed traffic capture (bench reports null)")
    units = d["units"]
    assert abs(bench.profiled_traffic(units) - d["verify_tc_kernel_dram_bytes"] - d["finalize_kernel_dram_bytes"]) < 1.0
    assert abs(bench.profiled_traffic(2 * units) - 2 * bench.profiled_traffic(units)) < 1.0
    # The capture reads at least the algorithmic K + V bytes of its launch (512 B per token-head).
    assert d["dram_bytes_per_unit"] >= 512


def test_stale_capture_gives_no_traffic(monkeypatch, tmp_path):
    with open(bench.PROFILE_TRAFFIC) as f:
        d = json.load(f)
    d["kernel_src_sha"] = "0" * 16
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(d))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(p))
    assert bench.profiled_traffic(1000) is None
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "missing.json"))
    assert bench.profiled_traffic(1000) is None
