"""Small parity cases run in a fresh process against a given build of the library
(the bounds-checked one): every path against the oracle, and the device status word
clear after each (a skipped out-of-range access would set HC_ERR_BOUNDS).

    python tests/_bounds_cases.py PATH_TO_LIBRARY
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402
import torch  # noqa: E402

from hyper_connection_residual_read_gb300 import _lib as hc  # noqa: E402
from hyper_connection_residual_read_gb300 import synth  # noqa: E402
from oracle import hc_oracle as O  # noqa: E402


def main(path: str) -> None:
    hc.load(path)
    from _hc import EPS, alloc_out, assert_matches_oracle, dev_f32, dev_weights, gpu_read
    assert hc.hc_read_bounds_checked(), "not the bounds-checked build"
    hc.hc_read_init(0, 2048, EPS)
    w = synth.make_weights(0)
    W = dev_weights(w)

    def check(label, got, want):
        assert_matches_oracle(got, want)
        code = hc.hc_read_status()
        assert code == hc.HC_OK, (label, code)
        print("ok", label, flush=True)

    cases = [(hc.HC_PATH_DECODE, 1, False), (hc.HC_PATH_DECODE, 4, True),
             (hc.HC_PATH_DECODE, 8, True), (hc.HC_PATH_DECODE, 13, True),
             (hc.HC_PATH_DECODE, 40, True), (hc.HC_PATH_DECODE_ONE_KERNEL, 4, True),
             (hc.HC_PATH_PREFILL, 8, True), (hc.HC_PATH_PREFILL, 129, False),
             (hc.HC_PATH_PREFILL, 300, True), (hc.HC_PATH_PREFILL_UNFUSED, 129, True),
             # several down tiles per CTA (the rings wrap across tiles), an 80-token
             # last tile
             (hc.HC_PATH_PREFILL, 2000, True)]
    for path, T, with_P in cases:
        a = synth.make_activations(600 + T, T, with_P)
        got = gpu_read(T, dev_f32(a["R"]), dev_f32(a["P"]), W, dev_f32(a["Rmix"]), path)
        want = O.hc_read(a["R"], a["P"], w["w_norm"], w["W_down"], w["W_up"], a["Rmix"], EPS)
        check(f"path {path} T {T} P {with_P}", got, want)

    # the y read-out, and the up stage run again on the read's lo
    T = 129
    a = synth.make_activations(650, T, True)
    R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
    shape = (T, synth.WIDTH)
    oy = [torch.empty(shape, dtype=torch.float32, device="cuda"),
          torch.empty(shape, dtype=torch.int16, device="cuda"),
          torch.empty(shape, dtype=torch.int16, device="cuda")]
    hc.hc_read_y(T, R, P, W["w_norm"], W["W_down"], W["W_up"], *oy)
    torch.cuda.synchronize()
    got = (oy[0].cpu().numpy(), oy[1].cpu().numpy().view(np.uint16), oy[2].cpu().numpy().view(np.uint16))
    check("y read-out", got, O.hc_read_y(a["R"], a["P"], w["w_norm"], w["W_down"], w["W_up"], EPS))
    ref = gpu_read(T, R, P, W, M, hc.HC_PATH_PREFILL)
    o = alloc_out(T)
    hc.hc_read_upmix(hc.HC_PATH_PREFILL, T, R, P, W["W_up"], M, *o)
    torch.cuda.synchronize()
    for x, y in zip(ref, (o[0].cpu().numpy(), o[1].cpu().numpy().view(np.uint16),
                          o[2].cpu().numpy().view(np.uint16))):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    assert hc.hc_read_status() == hc.HC_OK
    print("ok upmix rerun", flush=True)

    # the allocation-free entry
    T = 17
    a = synth.make_activations(660, T, True)
    o = alloc_out(T)
    hc.hc_read_noalloc(T, dev_f32(a["R"]), dev_f32(a["P"]), W["w_norm"], W["W_down"], W["W_up"],
                       dev_f32(a["Rmix"]), *o, eps=EPS)
    torch.cuda.synchronize()
    got = (o[0].cpu().numpy(), o[1].cpu().numpy().view(np.uint16), o[2].cpu().numpy().view(np.uint16))
    check("noalloc T 17", got,
          O.hc_read(a["R"], a["P"], w["w_norm"], w["W_down"], w["W_up"], a["Rmix"], EPS))
    print("all cases passed", flush=True)


if __name__ == "__main__":
    main(sys.argv[1])
