"""The GPU parity suites again with the one-CTA GEMM variant selected.

The CTA-pair kernels are the default; LMHEAD_GEMM=single selects the one-CTA
tcgen05 kernels (128 x 256 tiles), which share the epilogues and must give
the same results.  A few parity tests cover that variant directly; here the
parity, shard and autograd suites run in a child process with it selected
(tests that pick a variant themselves keep their choice).
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITE = ["tests/test_gpu_parity.py", "tests/test_gpu_shards.py", "tests/test_gpu_autograd.py"]


def test_parity_suites_pass_on_the_one_cta_variant():
    env = dict(os.environ, LMHEAD_GEMM="single")
    r = subprocess.run([sys.executable, "-m", "pytest", *SUITE, "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
