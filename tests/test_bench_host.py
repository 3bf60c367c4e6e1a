"""Host checks of bench.py's bookkeeping (no GPU): the DRAM-traffic record is
used only for the workload and kernel sources it was captured on."""

import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _record():
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        return json.load(f)


def test_traffic_record_matches_only_its_own_workload():
    rec = _record()
    cfg = dict(rec["config"])
    if rec["source_sha256"] == bench.kernel_source_digest():
        got = bench.recorded_traffic("gemm_dw", cfg)
        assert got is not None and got["dram_bytes_per_launch"] > 0
    for key, other in (("rows", "block-sparse tiles"), ("mode", "fwd"), ("keep_mask", "off"),
                       ("entropy", "metric-only"), ("N", 1024)):
        assert bench.recorded_traffic("gemm_dw", dict(cfg, **{key: other})) is None, key


def test_traffic_record_is_dropped_when_the_sources_change(monkeypatch):
    rec = _record()
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: "0" * 64)
    assert bench.recorded_traffic("gemm_dw", dict(rec["config"])) is None
