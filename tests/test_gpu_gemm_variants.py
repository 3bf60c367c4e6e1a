"""The GPU parity suites again with every contraction on one GEMM variant.

By default dHidden and dW run on CTA pairs with 256 x 512 tiles and the
projections on CTA pairs with 256 x 256 tiles.  LMHEAD_GEMM=single, =pair or
=wide puts all four contractions on the one-CTA (128 x 256 tiles), CTA-pair
(256 x 256) or wide CTA-pair (256 x 512) kernel; they share the epilogues and
must give the same results.  A few parity tests pick a variant
directly; here the parity, shard and autograd suites run in a child process
with each variant selected (tests that pick a variant themselves keep their
choice).
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITE = ["tests/test_gpu_parity.py", "tests/test_gpu_shards.py", "tests/test_gpu_autograd.py"]


@pytest.mark.parametrize("variant", ["single", "pair", "wide"])
def test_parity_suites_pass_on_one_variant(variant):
    env = dict(os.environ, LMHEAD_GEMM=variant)
    r = subprocess.run([sys.executable, "-m", "pytest", *SUITE, "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider"],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
