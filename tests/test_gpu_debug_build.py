"""The GPU test suite against the LMHEAD_DEBUG build of the library.

That build (liblmhead_debug.so, made by build()) checks every index its
kernels derive from data before the access it guards, and records
LMHEAD_EBOUNDS in the device status word instead of touching memory outside an
array, so a wrong index becomes a failed status check rather than a stray
access.
The suite runs in a child process with LMHEAD_LIBRARY=debug; its tests assert a
clean device status after their calls and compare with the oracle, so a
failed index check fails them.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITE = ["tests/test_gpu_parity.py", "tests/test_gpu_shards.py", "tests/test_gpu_sls.py",
         "tests/test_gpu_autograd.py", "tests/test_gpu_runtime.py"]


@pytest.fixture(scope="module", autouse=True)
def _debug_library():
    # build() makes it; build it here too if it is missing or stale
    from sft_keep_mask_gb300 import build as b
    b.build(debug=True)


def _env():
    return dict(os.environ, LMHEAD_LIBRARY="debug")


def test_the_debug_library_is_the_one_loaded():
    r = subprocess.run([sys.executable, "-c",
                        "from sft_keep_mask_gb300 import lmhead as L; "
                        "print(L.library_path()); print(L.lmhead_version())"],
                       env=_env(), cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert "liblmhead_debug.so" in r.stdout and "debug index checks" in r.stdout


def test_gpu_suite_passes_with_device_index_checks():
    r = subprocess.run([sys.executable, "-m", "pytest", *SUITE, "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider"],
                       env=_env(), cwd=ROOT, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
