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


def test_reference_arm_prints_the_contract_line():
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == line["value"] and cpu["cores"] >= 1
    # exactly the GPU arm's config object; the sample size is reported beside it
    import argparse
    args = argparse.Namespace(workload="tiny", chunk_rows=0, mode="fwdbwd", keep_off=False,
                              blocksparse=False)
    cfg = line["config"]
    assert cfg == bench.run_config(args, cfg["N"], cfg["H"], cfg["V"], cfg["kept_rows"], 1, True)
    assert line["sample_rows_per_step"] == min(32, cfg["kept_rows"])  # --ref-rows default


def test_clock_summary_reads_clocks_reasons_and_power():
    # nvidia-smi csv lines: index, clocks.sm, clocks.max.sm, power.draw, the
    # active reasons bitmask, then hw_slowdown, hw_thermal_slowdown,
    # sw_thermal_slowdown and sw_power_cap as Active / Not Active
    s = bench.ClockSampler(0)
    s.lines = [
        "0, 1500, 2070, 1350.5, 0x4, Not Active, Not Active, Not Active, Active\n",
        "0, 1540, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active\n",
        "0, 1520, 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active\n",
        "garbage\n",
    ]
    got = s.summary()
    assert got["sm_mhz"] == 1520 and got["sm_max_mhz"] == 2070 and got["samples"] == 3
    assert got["reasons"] == ["sw_power_cap"]
    assert got["power_w"] == (1350.5 + 1390.0) / 2  # the unreadable power sample is skipped
    empty = bench.ClockSampler(0)
    empty.lines = []
    assert empty.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                               "samples": 0, "power_w": None}
