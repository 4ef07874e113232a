"""GPU parity of the read on the edges of its input domain, against the CPU oracle.

The read is defined for any fp32 residual: the RMS norm is per (token, stream) and
scale-free up to eps ("#315 hc: the multi-token hyper-connection read split finer",
"What changes"), and the up projection, gate and mix run on whatever the chunk holds
("#1370 prefill: opt-in STRATA_HC_UPMIX=1 on CUDA ...", "What it does"). Every path
must therefore match the oracle on:

* residuals (and pending writes) scaled by powers of two from 2^-20 to 2^17: at
  2^-20 the outputs sit in fp16's subnormal range, at 2^17 some exceed fp16's
  largest finite value and their fp16 image must be infinite (the bf16 image stays
  finite); at 2^8 the output is 2^8 times the unscaled one (eps is negligible there);
* an all-zero stream (its rs is 1/sqrt(eps)) and a constant stream;
* a saturated gate: weights built so that every |u| lies between about 14 and 124,
  past the point where exp(-u) overflows fp32, with one stream always open so that
  no output is the sum of vanishing terms only.

Paths: the decode kernels, the one-kernel decode read, the tensor-core tile path
fused and unfused, and the 2560-wide read-out.
"""
import numpy as np
import pytest
import torch

import hyper_connection_residual_read_gb300 as hc
from hyper_connection_residual_read_gb300 import synth
from oracle import hc_oracle as O

from _hc import (EPS, MAX_TOKENS, TOL_F32, assert_matches_oracle, dev_f32,
                 dev_weights, gpu_read, rel_diff)

pytestmark = pytest.mark.gpu

# (path, tokens): the decode kernels at a few tokens, the tile path across a partial
# second tile
READ_PATHS = [(hc.HC_PATH_DECODE, 3), (hc.HC_PATH_DECODE_ONE_KERNEL, 4),
              (hc.HC_PATH_PREFILL, 200), (hc.HC_PATH_PREFILL_UNFUSED, 200)]
PATH_IDS = ["decode", "one_kernel", "prefill", "prefill_unfused"]
SCALES = [-20, -12, -6, 8, 17]


@pytest.fixture(scope="module")
def ctx():
    hc.hc_read_init(0, MAX_TOKENS, EPS)
    yield
    torch.cuda.synchronize()


@pytest.fixture(scope="module")
def weights(ctx):
    w = synth.make_weights(0)
    return w, dev_weights(w)


def _bf16(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def scaled(a: dict, k: int) -> dict:
    """R and P times 2^k (exact in fp32 over the range used here)."""
    f = np.float32(2.0 ** k)
    return {"R": a["R"] * f, "P": None if a["P"] is None else a["P"] * f, "Rmix": a["Rmix"]}


def read_and_oracle(w, W, a, T, path):
    got = gpu_read(T, dev_f32(a["R"]), dev_f32(a["P"]), W, dev_f32(a["Rmix"]), path)
    assert hc.hc_read_status() == 0
    want = O.hc_read(a["R"], a["P"], w["w_norm"], w["W_down"], w["W_up"], a["Rmix"], EPS)
    return got, want


@pytest.mark.parametrize("k", SCALES)
@pytest.mark.parametrize("path,T", READ_PATHS, ids=PATH_IDS)
def test_scaled_residual(weights, path, T, k):
    w, W = weights
    a = scaled(synth.make_activations(400 + T + k, T, True), k)
    got, want = read_and_oracle(w, W, a, T, path)
    assert_matches_oracle(got, want)
    if k == 17:
        # some outputs overflow fp16 (their image is +-inf); bf16 stays finite
        h = got[2]
        assert np.any((h & 0x7FFF) == 0x7C00)
        assert not np.any((got[1] & 0x7F80) == 0x7F80)
    if k == -20:
        # fp16 images in the subnormal range
        h = got[2] & 0x7FFF
        assert np.mean((h > 0) & (h < 0x0400)) > 0.5


@pytest.mark.parametrize("path,T", READ_PATHS, ids=PATH_IDS)
def test_power_of_two_scaling(weights, path, T):
    """read(2^8 R, 2^8 P) = 2^8 read(R, P) to the tolerance: eps is negligible next to
    the mean square at this scale, and every other step is linear or scale-free."""
    w, W = weights
    a = synth.make_activations(450 + T, T, True)
    base = gpu_read(T, dev_f32(a["R"]), dev_f32(a["P"]), W, dev_f32(a["Rmix"]), path)
    b = scaled(a, 8)
    up = gpu_read(T, dev_f32(b["R"]), dev_f32(b["P"]), W, dev_f32(b["Rmix"]), path)
    assert rel_diff(up[0] / np.float32(256.0), base[0]) <= TOL_F32


@pytest.mark.parametrize("path,T", READ_PATHS, ids=PATH_IDS)
def test_zero_and_constant_streams(weights, path, T):
    w, W = weights
    a = synth.make_activations(470 + T, T, True)
    a["R"][:, 1, :] = 0.0
    a["P"][:, 1, :] = 0.0
    a["R"][:, 2, :] = 0.75
    a["P"][:, 2, :] = 0.0
    got, want = read_and_oracle(w, W, a, T, path)
    assert_matches_oracle(got, want)


def saturating_case(seed: int, T: int):
    """Weights and inputs whose up projection saturates the gate: W_down rows all
    0.01 and a positive residual make every lo about 99; W_up row i is v_i / 320 in
    every column, |v_i| in [0.15, 1.25], so u_i = lo * v_i lies in about +-[14, 124].
    Stream 0 has v > 0 (its gate is open), the other streams mixed signs."""
    g = np.random.default_rng(seed)
    w = synth.make_weights(0)
    v = g.uniform(0.15, 1.25, 10240) * np.where(g.random(10240) < 0.5, -1.0, 1.0)
    v[:2560] = np.abs(v[:2560])
    w = {"w_norm": w["w_norm"], "W_down": _bf16(np.full((320, 10240), 0.01)),
         "W_up": _bf16(np.repeat((v / 320.0)[:, None], 320, axis=1))}
    a = synth.make_activations(seed, T, True)
    a["R"] = (0.75 + 0.5 * np.abs(g.standard_normal((T, 4, 2560)))).astype(np.float32)
    return w, a


@pytest.mark.parametrize("path,T", READ_PATHS, ids=PATH_IDS)
def test_saturated_gate(ctx, path, T):
    w, a = saturating_case(480 + T, T)
    st = O.hc_read(a["R"], a["P"], w["w_norm"], w["W_down"], w["W_up"], a["Rmix"], EPS,
                   stages=True)
    u = np.abs(st["u"])
    assert u.min() > 10 and u.max() > 100     # the construction does what it says
    got, want = read_and_oracle(w, dev_weights(w), a, T, path)
    assert_matches_oracle(got, want)


def _read_y(T, a, W):
    shape = (T, synth.WIDTH)
    o = (torch.empty(shape, dtype=torch.float32, device="cuda"),
         torch.empty(shape, dtype=torch.int16, device="cuda"),
         torch.empty(shape, dtype=torch.int16, device="cuda"))
    hc.hc_read_y(T, dev_f32(a["R"]), dev_f32(a["P"]), W["w_norm"], W["W_down"], W["W_up"], *o)
    torch.cuda.synchronize()
    assert hc.hc_read_status() == 0
    return (o[0].cpu().numpy(), o[1].cpu().numpy().view(np.uint16),
            o[2].cpu().numpy().view(np.uint16))


@pytest.mark.parametrize("case", ["scale-12", "scale17", "zero_constant", "saturated"])
def test_readout_y_edges(weights, case):
    T = 200
    w, W = weights
    if case == "saturated":
        w, a = saturating_case(490, T)
        W = dev_weights(w)
    else:
        a = synth.make_activations(491, T, True)
        if case == "zero_constant":
            a["R"][:, 1, :] = 0.0
            a["P"][:, 1, :] = 0.0
            a["R"][:, 2, :] = 0.75
            a["P"][:, 2, :] = 0.0
        else:
            a = scaled(a, int(case[5:]))
    got = _read_y(T, a, W)
    want = O.hc_read_y(a["R"], a["P"], w["w_norm"], w["W_down"], w["W_up"], EPS)
    assert_matches_oracle(got, want)


def test_decode_and_tile_path_agree_on_a_wide_range(weights):
    """One input whose tokens span 2^-20 .. 2^17 in scale: the decode kernels (chunks of
    8) and the tile path each match the oracle token by token."""
    w, W = weights
    T = 12
    a = synth.make_activations(495, T, True)
    ks = np.linspace(-20, 17, T).round().astype(int)
    f = (2.0 ** ks).astype(np.float32)[:, None, None]
    a["R"] = a["R"] * f
    a["P"] = a["P"] * f
    want = O.hc_read(a["R"], a["P"], w["w_norm"], w["W_down"], w["W_up"], a["Rmix"], EPS)
    for path in (hc.HC_PATH_DECODE, hc.HC_PATH_PREFILL):
        got = gpu_read(T, dev_f32(a["R"]), dev_f32(a["P"]), W, dev_f32(a["Rmix"]), path)
        assert hc.hc_read_status() == 0
        for t in range(T):   # each token against its own scale
            assert_matches_oracle(tuple(x[t:t + 1] for x in got), tuple(x[t:t + 1] for x in want))
