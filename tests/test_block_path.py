"""The 128-token block path (pair transitions, affine block scan, block output).

It serves the gated delta rule at dk = dv = 128 when GDN_BLOCK_PATH=1 is set
before the library is first used, so the whole parity suite is run again in
a child process with the switch on: every case there compares against the
fp64 oracle with the same tolerances.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_suite_on_the_block_path(cuda_lib):
    env = dict(os.environ, GDN_BLOCK_PATH="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_parity.py"),
                        os.path.join(ROOT, "tests", "test_prologue.py"), "-q", "-x", "-m", "gpu",
                        "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
