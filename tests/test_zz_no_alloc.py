"""The allocation-free entry point, hc_read_noalloc, against hc_read.

Callers that cannot allocate device memory (plug-ins inside an engine that owns
all device memory, loops that must not synchronise the device, callers that never
run hc_read_init) use hc_read_noalloc, whose scratch is a fixed device array in
the library. This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh
process.
"""
import numpy as np
import pytest
import torch

import hyper_connection_residual_read_gb300 as hc
from hyper_connection_residual_read_gb300 import synth

from _hc import (EPS, MAX_TOKENS, TOL_F32, alloc_out, assert_images_close, dev_f32,
                 dev_weights, gpu_read, rel_diff)

pytestmark = pytest.mark.gpu


def test_noalloc_matches_hc_read_on_consecutive_calls():
    hc.hc_read_init(0, MAX_TOKENS, EPS)          # for the reference entry point only
    w = synth.make_weights(0)
    W = dev_weights(w)
    for call, (T, with_P) in enumerate([(5, True), (8, False)]):   # two calls in a row
        a = synth.make_activations(700 + call, T, with_P)
        R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
        want = gpu_read(T, R, P, W, M)
        o = alloc_out(T)
        hc.hc_read_noalloc(T, R, P, W["w_norm"], W["W_down"], W["W_up"], M, *o, eps=EPS)
        torch.cuda.synchronize()
        got = (o[0].cpu().numpy(), o[1].cpu().numpy().view(np.uint16),
               o[2].cpu().numpy().view(np.uint16))
        assert rel_diff(got[0], want[0]) <= TOL_F32
        # same criterion as against the oracle: within 1 ulp, or within the fp32 band
        delta = TOL_F32 * float(np.max(np.abs(want[0].astype(np.float64))))
        assert_images_close(got[1], want[1], want[0], "bf16", delta)
        assert_images_close(got[2], want[2], want[0], "fp16", delta)


def test_noalloc_refuses_more_than_its_scratch_holds():
    w = synth.make_weights(0)
    W = dev_weights(w)
    a = synth.make_activations(710, 65, False)
    o = alloc_out(65)
    with pytest.raises(hc.HcReadError) as e:
        hc.hc_read_noalloc(65, dev_f32(a["R"]), None, W["w_norm"], W["W_down"], W["W_up"],
                           dev_f32(a["Rmix"]), *o, eps=EPS)
    assert e.value.code == -1
