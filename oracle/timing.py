"""Timing helper for the CPU baseline of the prefill chunks: the oracle read of one
set of tokens, timed in the process that runs it.

TEST INFRASTRUCTURE ONLY, like the oracle itself: only the ``cpu_baseline`` leg of
``bench.py`` uses it, from processes it starts with the spawn method (a worker
function has to live in an importable module for that).
"""
import time

from . import hc_oracle as O


def timed_read(args) -> float:
    """args = (R, Rmix, weights dict, eps); the read without a pending write. Returns
    the seconds the oracle took."""
    R, Rmix, w, eps = args
    t0 = time.perf_counter()
    O.hc_read(R, None, w["w_norm"], w["W_down"], w["W_up"], Rmix, eps)
    return time.perf_counter() - t0
