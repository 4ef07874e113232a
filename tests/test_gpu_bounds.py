"""The bounds-checked build (-DHC_BOUNDS_CHECK) on the small parity cases.

It stands in for a memory checker: every hand-indexed global access of every kernel
is first checked against its buffer's extent as the kernel's arguments give it, and
an access out of range is skipped and reported through the device status word
(HC_ERR_BOUNDS) instead of trapping. The variant is built on demand and run in a fresh
process (the binding loads one library per process): every decode, one-kernel, tile
path, y read-out, stage re-run and allocation-free case matches the oracle, and the
status word stays clear after each.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_parity_cases_under_the_bounds_checked_build():
    from hyper_connection_residual_read_gb300 import build
    path = build.build_bounds_checked()
    r = subprocess.run([sys.executable, os.path.join(HERE, "_bounds_cases.py"), path],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "all cases passed" in r.stdout
