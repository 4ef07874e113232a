"""Failure detection on the GPU, made without a GPU fault.

The one-kernel decode read waits inside the kernel for every CTA's part of lo, with
a bound ("#2226 STRATA_HC_PERSIST=1 (opt-in, HIP): the verifier's hyper-connection
read as one persistent kernel", "What changed": a barrier timeout, then the read
falls back instead of hanging). A test shortens that bound through the library's
internal entry so that the wait runs out: the call returns, the device status word
reports HC_ERR_TIMEOUT, and the next read, with the bound restored, gives the bits
of a read made before. Only that wait is shortened: it spins on a counter in global
memory and has no copy in flight, so running out of it faults nothing.
"""
import numpy as np
import pytest
import torch

import hyper_connection_residual_read_gb300 as hc
from hyper_connection_residual_read_gb300 import synth

from _hc import EPS, alloc_out, dev_f32, dev_weights, gpu_read

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def weights():
    hc.hc_read_init(0, 64, EPS)
    w = synth.make_weights(0)
    yield w, dev_weights(w)
    hc.hc_read_set_wait_limit(0)
    torch.cuda.synchronize()


def test_one_kernel_wait_runs_out_and_reports_a_timeout(weights):
    w, W = weights
    T = 4
    a = synth.make_activations(810, T, True)
    R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
    ref = gpu_read(T, R, P, W, M, hc.HC_PATH_DECODE_ONE_KERNEL)
    ref2 = gpu_read(T, R, P, W, M, hc.HC_PATH_DECODE)
    assert hc.hc_read_status() == hc.HC_OK
    hc.hc_read_set_wait_limit(1)            # 1 ns: a CTA that has to wait gives up
    codes = []
    for _ in range(5):
        o = alloc_out(T)
        hc.hc_read_path(hc.HC_PATH_DECODE_ONE_KERNEL, T, R, P, W["w_norm"], W["W_down"],
                        W["W_up"], M, *o)
        torch.cuda.synchronize()
        codes.append(hc.hc_read_status())
        if codes[-1] == hc.HC_ERR_TIMEOUT:
            break
    assert codes[-1] == hc.HC_ERR_TIMEOUT, codes
    assert hc.hc_read_status() == hc.HC_OK          # the status word was cleared
    hc.hc_read_set_wait_limit(0)                    # back to 2 s
    for path, want in ((hc.HC_PATH_DECODE_ONE_KERNEL, ref), (hc.HC_PATH_DECODE, ref2)):
        got = gpu_read(T, R, P, W, M, path)
        for x, y in zip(want, got):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    assert hc.hc_read_status() == hc.HC_OK
