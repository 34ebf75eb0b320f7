"""bench.py's host logic: the committed DRAM-traffic capture is used only while the verify call's
sources are the ones it was taken on, only for a call whose kernels it holds, and it scales with
the units a launch processes."""

import json

import pytest

import bench


def _capture():
    with open(bench.PROFILE_TRAFFIC) as f:
        return json.load(f)


def test_committed_traffic_matches_current_sources():
    d = _capture()
    if d["kernel_src_sha"] != bench.kernel_source_sha():
        pytest.skip("the verify sources changed since the committed traffic capture (bench reports null)")
    units = d["units"]
    kernels = d["calls"]["ssd_verify_select"]
    want = sum(d["kernel_dram_bytes"][k] for k in kernels)
    assert abs(bench.profiled_traffic(units, "ssd_verify_select") - want) < 1.0
    assert abs(bench.profiled_traffic(2 * units) - 2 * bench.profiled_traffic(units)) < 1.0
    # The capture reads at least the algorithmic K + V bytes of its launch (512 B per token-head).
    assert want / units >= 512


def test_stale_or_incomplete_capture_gives_no_traffic(monkeypatch, tmp_path):
    d = _capture()
    d["kernel_src_sha"] = bench.kernel_source_sha()
    d["kernel_dram_bytes"] = {"verify_tc_kernel": 600.0 * d["units"], "crit_select_kernel": 50.0 * d["units"]}
    d["calls"] = {"ssd_verify_select": ["verify_tc_kernel", "crit_select_kernel"],
                  "ssd_verify_attn": ["verify_tc_kernel", "finalize_kernel"]}
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(d))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(p))
    assert abs(bench.profiled_traffic(1000, "ssd_verify_select") - 650.0 * 1000) < 1e-6
    # finalize_kernel is not in the capture: no number for ssd_verify_attn, nor for an unknown call.
    assert bench.profiled_traffic(1000, "ssd_verify_attn") is None
    assert bench.profiled_traffic(1000, "ssd_draft_attn") is None
    d["kernel_src_sha"] = "0" * 16
    p.write_text(json.dumps(d))
    assert bench.profiled_traffic(1000) is None
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "missing.json"))
    assert bench.profiled_traffic(1000) is None
