"""Host checks of the persistent GEMMs' work schedule, no GPU needed.

``tests/host/schedule_check.cu`` includes the kernels' own scheduling helpers
(tile raster, chunk spans, the plain / split-tail work schedule) and runs them
on the CPU: every tile index must map to a distinct tile of the grid, the
chunks must cover the kept rows in order, every worker's segments together
must cover every (tile, K block) once, the split tail in at most max_split
parts per tile (slots in K order, faster than unsplit), and the
512-column tiles of the CTA-pair kernel must cover every 256-column tile once,
counted and ordered as the dHidden reduction counts and orders them.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_schedule_helpers_cover_every_tile_and_row(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "schedule_check"
    src = os.path.join(ROOT, "tests", "host", "schedule_check.cu")
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                        "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-o",
                        str(exe), src], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
