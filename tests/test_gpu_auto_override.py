"""The HC_READ_DECODE_MAX_T override of HC_PATH_AUTO's crossover: each setting runs in
a fresh process (hc_read_init reads the variable). 64 and 0 move the crossover; a
malformed value keeps the default of 48."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("value,crossover", [("64", 64), ("0", 0), ("4x", 48)])
def test_auto_crossover_follows_the_environment(value, crossover):
    env = dict(os.environ, HC_READ_DECODE_MAX_T=value)
    r = subprocess.run([sys.executable, os.path.join(HERE, "_auto_override_case.py"),
                        str(crossover)], capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "all cases passed" in r.stdout
