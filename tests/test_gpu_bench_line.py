"""bench.py on a small workload: the JSON line carries every key of its
contract, with values that hang together (device-timed value, end-to-end
rate through host buffers, dominant-kernel roofline, CPU oracle baseline,
launch count, clock record, forward / backward split of the step)."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_fwd_bwd_line_has_the_contract_keys():
    line = _bench("--workload", "qwen3_4b", "--rows", "4096", "--steps", "3", "--warmup", "3",
                  "--cpu-rows", "8")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "cpu_baseline", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["dtype"] == "bf16" and line["vs_baseline"] is None
    assert line["device_status"] == 0
    cfg = line["config"]
    assert cfg["workload"] == "qwen3_4b" and cfg["N"] == 4096 and cfg["mode"] == "fwdbwd"
    nk = cfg["kept_rows"]
    assert 0 < nk <= cfg["N"]
    # value = kept rows per second of device time
    assert line["value"] == pytest.approx(nk / (line["ms_per_step"] / 1e3), rel=1e-6)
    # TFLOP/s counted with the backward's recompute (8 Nk H V) and without it
    flops = 8.0 * nk * cfg["H"] * cfg["V"]
    assert line["tflops"] == pytest.approx(flops / (line["ms_per_step"] / 1e3) / 1e12, rel=1e-6)
    assert line["tflops_recompute_free"] == pytest.approx(0.75 * line["tflops"], rel=1e-6)
    # the forward and backward parts of the median step add up to about a step
    parts = line["pass_ms"]
    assert parts["fwd"] > 0 and parts["bwd"] > parts["fwd"]
    assert parts["fwd"] + parts["bwd"] == pytest.approx(line["step_ms"]["median"], rel=0.25)
    roof = line["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert roof["kernel"] in ("gemm_fwd", "gemm_dz", "gemm_dh", "gemm_dw")
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], rel=1e-9)
    assert roof["traffic"] is None  # no capture of this workload is on record
    e2e = line["e2e"]
    assert e2e["unit"] == line["unit"] and e2e["value"] > 0
    assert e2e["h2d_bytes_per_step"] > cfg["N"] * cfg["H"] * 2  # at least the hidden states
    assert e2e["d2h_bytes_per_step"] == 2 * cfg["N"] * 4       # logprob and entropy
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] > 0 and cpu["cores"] >= 1
    assert cpu["sample"].startswith("8 kept rows")
    # every library kernel of the timed steps was counted, and the GEMMs ran
    assert line["gpu_launches"] >= 3 * 8
    assert line["kernels"]["gemm_dh"]["launches"] >= 3
    clk = line["clocks"]
    assert clk["sm_max_mhz"] > 0 and isinstance(clk["reasons"], list)


def test_forward_only_line():
    line = _bench("--workload", "qwen3_4b", "--rows", "4096", "--mode", "fwd", "--steps", "3",
                  "--warmup", "3", "--no-e2e", "--no-cpu-baseline")
    cfg = line["config"]
    assert cfg["mode"] == "fwd" and line["device_status"] == 0
    assert line["pass_ms"]["bwd"] is None
    assert line["roofline"]["kernel"] == "gemm_fwd"
    flops = 2.0 * cfg["kept_rows"] * cfg["H"] * cfg["V"]
    assert line["tflops"] == pytest.approx(flops / (line["ms_per_step"] / 1e3) / 1e12, rel=1e-6)
    assert line["tflops_recompute_free"] == pytest.approx(line["tflops"], rel=1e-6)
    assert line["e2e"] is None and line["cpu_baseline"] is None
