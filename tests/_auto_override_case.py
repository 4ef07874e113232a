"""HC_PATH_AUTO under the HC_READ_DECODE_MAX_T override, run in a fresh process whose
environment sets it (hc_read_init reads it): the automatic path must give the bits of
the decode path at and below the given count and those of the tile path above it.

    HC_READ_DECODE_MAX_T=N python tests/_auto_override_case.py EXPECTED_CROSSOVER
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402

from hyper_connection_residual_read_gb300 import _lib as hc  # noqa: E402
from hyper_connection_residual_read_gb300 import synth  # noqa: E402


def main(crossover: int) -> None:
    from _hc import EPS, dev_f32, dev_weights, gpu_read
    hc.hc_read_init(0, 128, EPS)
    W = dev_weights(synth.make_weights(5))

    def same(x, y):
        return all(np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                                  b.view(np.uint32) if b.dtype == np.float32 else b)
                   for a, b in zip(x, y))

    for T in sorted({t for t in (1, crossover, crossover + 1) if 1 <= t <= 128}):
        a = synth.make_activations(700 + T, T, True)
        R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
        auto = gpu_read(T, R, P, W, M)
        dec = gpu_read(T, R, P, W, M, hc.HC_PATH_DECODE)
        tile = gpu_read(T, R, P, W, M, hc.HC_PATH_PREFILL)
        want, other = (dec, tile) if T <= crossover else (tile, dec)
        assert same(auto, want), (T, crossover)
        # the two paths differ in rounding, so the check above tells them apart
        assert not same(auto, other), (T, crossover)
        assert hc.hc_read_status() == hc.HC_OK
        print("ok T", T, flush=True)
    print("all cases passed", flush=True)


if __name__ == "__main__":
    main(int(sys.argv[1]))
