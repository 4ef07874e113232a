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

from oracle import hc_oracle as O

from _hc import EPS, MAX_TOKENS, alloc_out, assert_matches_oracle, dev_f32, dev_weights, gpu_read

pytestmark = pytest.mark.gpu


def test_noalloc_matches_hc_read_on_consecutive_calls():
    """Calls in a row, with and without a pending write, over token counts that use one
    to eight 8-token chunks of the fixed array (64 tokens reach its last slot): the
    outputs are bitwise those of hc_read on the same decode kernels, and match the
    oracle."""
    hc.hc_read_init(0, MAX_TOKENS, EPS)          # for the reference entry point only
    w = synth.make_weights(0)
    W = dev_weights(w)
    for call, (T, with_P) in enumerate([(5, True), (8, False), (13, True), (64, True),
                                        (64, False), (17, False)]):
        a = synth.make_activations(700 + call, T, with_P)
        R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
        want = gpu_read(T, R, P, W, M, hc.HC_PATH_DECODE)
        o = alloc_out(T)
        for x in o:
            x.fill_(-1)
        hc.hc_read_noalloc(T, R, P, W["w_norm"], W["W_down"], W["W_up"], M, *o, eps=EPS)
        torch.cuda.synchronize()
        got = (o[0].cpu().numpy(), o[1].cpu().numpy().view(np.uint16),
               o[2].cpu().numpy().view(np.uint16))
        for x, y in zip(want, got):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), (T, with_P)
        if T in (13, 64):
            oracle = O.hc_read(a["R"], a["P"], w["w_norm"], w["W_down"], w["W_up"], a["Rmix"],
                               EPS)
            assert_matches_oracle(got, oracle)


def test_noalloc_refuses_more_than_its_scratch_holds():
    w = synth.make_weights(0)
    W = dev_weights(w)
    a = synth.make_activations(710, 65, False)
    o = alloc_out(65)
    with pytest.raises(hc.HcReadError) as e:
        hc.hc_read_noalloc(65, dev_f32(a["R"]), None, W["w_norm"], W["W_down"], W["W_up"],
                           dev_f32(a["Rmix"]), *o, eps=EPS)
    assert e.value.code == -1
