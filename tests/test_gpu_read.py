"""GPU parity of the hyper-connection read against the CPU oracle, through the C ABI.

Cases follow the workloads of the decode verify window and prefill chunks:
one token without a pending write (seed 0), the verify-window sweep T = 1..8 with
and without the pending write (seeds 1..16, one per case), ragged token counts
that cross the 8-token launch chunks, a cold round of 48 weight sets, and long
prefill chunks checked on sampled tokens. Plus determinism, the pending-write
identity, argument errors and output guard bytes.
"""
import os

import numpy as np
import pytest
import torch

import hyper_connection_residual_read_gb300 as hc
from hyper_connection_residual_read_gb300 import synth
from oracle import hc_oracle as O

from _hc import (EPS, MAX_TOKENS, TOL_F32, alloc_out, assert_matches_oracle, dev_f32,
                 dev_u16, dev_weights, gpu_read, rel_diff)

pytestmark = pytest.mark.gpu

PATHS = [None, hc.HC_PATH_DECODE, hc.HC_PATH_DECODE_ONE_KERNEL]


@pytest.fixture(scope="module")
def ctx():
    hc.hc_read_init(0, MAX_TOKENS, EPS)
    yield
    torch.cuda.synchronize()


@pytest.fixture(scope="module")
def weights(ctx):
    w = synth.make_weights(0)
    return w, dev_weights(w)


def run_case(weights, T, with_P, seed, path=None):
    w, W = weights
    a = synth.make_activations(seed, T, with_P)
    got = gpu_read(T, dev_f32(a["R"]), dev_f32(a["P"]), W, dev_f32(a["Rmix"]), path)
    want = O.hc_read(a["R"], a["P"], w["w_norm"], w["W_down"], w["W_up"], a["Rmix"], EPS)
    return got, want


@pytest.mark.parametrize("path", PATHS)
def test_single_token_no_pending_write(weights, path):
    got, want = run_case(weights, 1, False, 0, path)
    assert_matches_oracle(got, want)


@pytest.mark.parametrize("T", range(1, 9))
@pytest.mark.parametrize("with_P", [False, True])
def test_verify_window_sweep(weights, T, with_P):
    seed = 1 + 2 * (T - 1) + int(with_P)          # seeds 1..16, one per case
    got, want = run_case(weights, T, with_P, seed)
    assert_matches_oracle(got, want)


@pytest.mark.parametrize("path", [hc.HC_PATH_DECODE, hc.HC_PATH_DECODE_ONE_KERNEL])
def test_chained_reads_wait_for_their_inputs(weights, path):
    """Three reads back to back on one stream, each taking the previous read's fp32
    output as its residual, with no synchronisation between them. The decode kernels
    start early (programmatic dependent launch) and may read only weights before
    the previous kernel has finished: a read that loaded its residual, its pending
    write, the mix or lo too soon would see a partly written or stale buffer. A
    read of other inputs first leaves a different lo in scratch."""
    w, W = weights
    for T in (1, 5, 8):
        other = synth.make_activations(900 + T, T, True)
        gpu_read(T, dev_f32(other["R"]), dev_f32(other["P"]), W, dev_f32(other["Rmix"]), path)
        acts = [synth.make_activations(910 + 3 * T + i, T, True) for i in range(3)]
        R = dev_f32(acts[0]["R"])
        Ps = [dev_f32(a["P"]) for a in acts]
        Ms = [dev_f32(a["Rmix"]) for a in acts]
        outs = [alloc_out(T) for _ in acts]
        torch.cuda.synchronize()
        for P, M, o in zip(Ps, Ms, outs):
            hc.hc_read_path(path, T, R, P, W["w_norm"], W["W_down"], W["W_up"], M, *o)
            R = o[0]
        torch.cuda.synchronize()
        r = acts[0]["R"]
        for a, o in zip(acts, outs):
            want = O.hc_read(r, a["P"], w["w_norm"], w["W_down"], w["W_up"], a["Rmix"], EPS)
            got = (o[0].cpu().numpy(), o[1].cpu().numpy().view(np.uint16),
                   o[2].cpu().numpy().view(np.uint16))
            assert_matches_oracle(got, want)
            r = got[0]


@pytest.mark.parametrize("T", [9, 13, 16, 17, 31])
@pytest.mark.parametrize("path", [hc.HC_PATH_DECODE, hc.HC_PATH_DECODE_ONE_KERNEL])
def test_ragged_token_counts(weights, T, path):
    got, want = run_case(weights, T, True, 100 + T, path)
    assert_matches_oracle(got, want)


@pytest.mark.parametrize("T,with_P", [(33, True), (40, False), (57, True), (64, True), (65, False),
                                      (130, True)])
def test_decode_passes_of_up_to_64_tokens(weights, T, with_P):
    """The decode kernels read up to 64 tokens in one pass over the weights (the down
    kernel in chunks of 5-8 tokens, the up kernel on all of them); 65 and 130 tokens
    take a second and third pass."""
    got, want = run_case(weights, T, with_P, 150 + T, hc.HC_PATH_DECODE)
    assert_matches_oracle(got, want)


@pytest.mark.parametrize("T", [1, 4, 8])
def test_one_kernel_decode_path(weights, T):
    got, want = run_case(weights, T, True, 300 + T, hc.HC_PATH_DECODE_ONE_KERNEL)
    assert_matches_oracle(got, want)


def test_bitwise_repeatable(weights):
    w, W = weights
    a = synth.make_activations(7, 8, True)
    R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
    first = gpu_read(8, R, P, W, M)
    for _ in range(5):
        again = gpu_read(8, R, P, W, M)
        for x, y in zip(first, again):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_pending_write_equals_preadded(weights):
    w, W = weights
    a = synth.make_activations(8, 5, True)
    pre = (a["R"] + a["P"]).astype(np.float32)
    x = gpu_read(5, dev_f32(a["R"]), dev_f32(a["P"]), W, dev_f32(a["Rmix"]))
    y = gpu_read(5, dev_f32(pre), None, W, dev_f32(a["Rmix"]))
    for p, q in zip(x, y):
        assert np.array_equal(p.view(np.uint8), q.view(np.uint8))


@pytest.mark.parametrize("path", [hc.HC_PATH_DECODE, hc.HC_PATH_DECODE_ONE_KERNEL])
def test_token_batch_invariance_decode(weights, path):
    """Token t's bits do not depend on the other tokens of the call (40 tokens in one
    pass of the decode kernels, 8 in the one-kernel read)."""
    w, W = weights
    n = 40 if path == hc.HC_PATH_DECODE else 8
    a = synth.make_activations(9, n, True)
    R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
    full = gpu_read(n, R, P, W, M, path)
    for t in (0, 5, 7) + ((13, 39) if n > 8 else ()):
        one = gpu_read(1, R[t:t + 1].contiguous(), P[t:t + 1].contiguous(), W,
                       M[t:t + 1].contiguous(), path)
        assert np.array_equal(one[0][0].view(np.uint32), full[0][t].view(np.uint32))


def test_zero_tokens_is_a_no_op(weights):
    w, W = weights
    o = alloc_out(1)
    o[0].fill_(3.0)
    a = synth.make_activations(1, 1, False)
    hc.hc_read(0, dev_f32(a["R"]), None, W["w_norm"], W["W_down"], W["W_up"],
               dev_f32(a["Rmix"]), *o)
    torch.cuda.synchronize()
    assert bool((o[0] == 3.0).all())


def test_output_guard_bytes_untouched(weights):
    w, W = weights
    T, G = 3, 4096
    a = synth.make_activations(10, T, True)
    n = T * 4 * 2560
    big = torch.full((n + 2 * G,), 7.0, dtype=torch.float32, device="cuda")
    b16 = torch.full((n + 2 * G,), 0x1234, dtype=torch.int16, device="cuda")
    h16 = torch.full((n + 2 * G,), 0x4321, dtype=torch.int16, device="cuda")
    hc.hc_read(T, dev_f32(a["R"]), dev_f32(a["P"]), W["w_norm"], W["W_down"], W["W_up"],
               dev_f32(a["Rmix"]), big[G:G + n], b16[G:G + n], h16[G:G + n])
    torch.cuda.synchronize()
    for buf, v in ((big, 7.0), (b16, 0x1234), (h16, 0x4321)):
        assert bool((buf[:G] == v).all()) and bool((buf[G + n:] == v).all())


def test_argument_errors_are_refused(weights):
    w, W = weights
    a = synth.make_activations(1, 2, True)
    R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
    o = alloc_out(2)
    args = dict(R=R, P=P, w_norm=W["w_norm"], W_down=W["W_down"], W_up=W["W_up"], Rmix=M,
                out_f32=o[0], out_bf16=o[1], out_fp16=o[2])

    def call(T=2, **kw):
        d = dict(args)
        d.update(kw)
        hc.hc_read(T, d["R"], d["P"], d["w_norm"], d["W_down"], d["W_up"], d["Rmix"],
                   d["out_f32"], d["out_bf16"], d["out_fp16"])

    bad = [
        dict(R=0),                                   # null
        dict(W_up=0),
        dict(out_fp16=0),
        dict(R=R.data_ptr() + 4),                    # misaligned
        dict(out_bf16=o[0]),                         # outputs overlap
        dict(out_f32=R),                             # output overlaps an input
        dict(R=torch.zeros(2, 4, 2560).data_ptr()),  # host memory
    ]
    for kw in bad:
        with pytest.raises(hc.HcReadError) as e:
            call(**kw)
        assert e.value.code == -1, kw
    with pytest.raises(hc.HcReadError):
        call(T=-1)
    with pytest.raises(hc.HcReadError):
        call(T=MAX_TOKENS + 1)
    with pytest.raises(hc.HcReadError):
        hc.hc_read_path(17, 2, R, P, W["w_norm"], W["W_down"], W["W_up"], M, *o)
    with pytest.raises(hc.HcReadError):
        hc.hc_read_path(-1, 2, R, P, W["w_norm"], W["W_down"], W["W_up"], M, *o)
    assert hc.hc_read_status() == 0


def test_cold_round_sampled(ctx):
    """48 weight sets (larger than L2) rotated over 96 reads of 4 tokens with a
    pending write; reads 0, 47 and 95 are checked against the oracle."""
    T = 4
    sets = [synth.make_weights(1000 + k) for k in range(48)]
    Wdev = [dev_weights(s) for s in sets]
    acts = [synth.make_activations(2000 + i, T, True) for i in range(96)]
    outs = [alloc_out(T) for _ in range(96)]
    for i in range(96):
        a, W = acts[i], Wdev[i % 48]
        hc.hc_read(T, dev_f32(a["R"]), dev_f32(a["P"]), W["w_norm"], W["W_down"], W["W_up"],
                   dev_f32(a["Rmix"]), *outs[i])
    torch.cuda.synchronize()
    for i in (0, 47, 95):
        w, a = sets[i % 48], acts[i]
        got = (outs[i][0].cpu().numpy(), outs[i][1].cpu().numpy().view(np.uint16),
               outs[i][2].cpu().numpy().view(np.uint16))
        want = O.hc_read(a["R"], a["P"], w["w_norm"], w["W_down"], w["W_up"], a["Rmix"], EPS)
        assert_matches_oracle(got, want)


@pytest.mark.parametrize("T,seed", [(8192, 100), (32768, 104)])
def test_prefill_chunk_sampled_tokens(weights, T, seed):
    """A long chunk in one call; the first and last 128 tokens and 256 random ones
    are checked against the oracle, plus NaN/Inf-free output everywhere."""
    w, W = weights
    a = synth.make_prefill_chunk(seed, T)
    R, M = dev_f32(a["R"]), dev_f32(a["Rmix"])
    o = alloc_out(T)
    hc.hc_read(T, R, None, W["w_norm"], W["W_down"], W["W_up"], M, *o)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(o[0]).all())
    rng = np.random.default_rng(seed)
    idx = np.unique(np.concatenate([np.arange(128), np.arange(T - 128, T),
                                    rng.choice(T, 256, replace=False)]))
    want = O.hc_read_tokens(idx, a["R"], None, w["w_norm"], w["W_down"], w["W_up"],
                            a["Rmix"], EPS)
    ti = torch.from_numpy(idx).cuda()
    got = (o[0][ti].cpu().numpy(), o[1][ti].cpu().numpy().view(np.uint16),
           o[2][ti].cpu().numpy().view(np.uint16))
    assert_matches_oracle(got, want)
    if T == 8192:
        # the unfused pair (up GEMM writing gated, then the mix) gives the same bits
        o2 = alloc_out(T)
        hc.hc_read_path(hc.HC_PATH_PREFILL_UNFUSED, T, R, None, W["w_norm"], W["W_down"],
                        W["W_up"], M, *o2)
        torch.cuda.synchronize()
        for x, y in zip(o, o2):
            assert bool(torch.equal(x, y))
    assert hc.hc_read_status() == 0


def test_prefill_several_tiles_per_cta_partial_last_tile(weights):
    """T = 2000 with P: 16 token tiles (256 down tiles over at most 152 CTAs, so CTAs
    take several, and the R and operand rings wrap across tiles), the last tile 80
    tokens long (R's rows past T are read as zero). The first and last 128 tokens and
    128 random ones against the oracle; the same bits from a second call."""
    w, W = weights
    T = 2000
    a = synth.make_activations(2000, T, True)
    R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
    o = alloc_out(T)
    hc.hc_read_path(hc.HC_PATH_PREFILL, T, R, P, W["w_norm"], W["W_down"], W["W_up"], M, *o)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(o[0]).all())
    rng = np.random.default_rng(2000)
    idx = np.unique(np.concatenate([np.arange(128), np.arange(T - 128, T),
                                    rng.choice(T, 128, replace=False)]))
    want = O.hc_read_tokens(idx, a["R"], a["P"], w["w_norm"], w["W_down"], w["W_up"],
                            a["Rmix"], EPS)
    ti = torch.from_numpy(idx).cuda()
    got = (o[0][ti].cpu().numpy(), o[1][ti].cpu().numpy().view(np.uint16),
           o[2][ti].cpu().numpy().view(np.uint16))
    assert_matches_oracle(got, want)
    o2 = alloc_out(T)
    hc.hc_read_path(hc.HC_PATH_PREFILL, T, R, P, W["w_norm"], W["W_down"], W["W_up"], M, *o2)
    torch.cuda.synchronize()
    for x, y in zip(o, o2):
        assert bool(torch.equal(x, y))
    assert hc.hc_read_status() == 0


def test_self_check_passes(ctx):
    code, rep = hc.hc_read_check(8, 1234)
    assert code == 0, rep
    assert rep["repeat_bitwise"] and rep["pending_write_bitwise"] and rep["images_bitwise"]
    assert rep["sm_count"] > 0


# ---------------------------------------------------------------------------
# the tensor-core tile path
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,with_P", [(1, False), (8, True), (9, True), (127, False),
                                      (128, True), (129, False), (300, True)])
def test_prefill_path_against_oracle(weights, T, with_P):
    got, want = run_case(weights, T, with_P, 200 + T, hc.HC_PATH_PREFILL)
    assert_matches_oracle(got, want)


def test_prefill_fused_equals_unfused_bitwise(weights):
    w, W = weights
    T = 300
    a = synth.make_activations(11, T, True)
    R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
    fused = gpu_read(T, R, P, W, M, hc.HC_PATH_PREFILL)
    unfused = gpu_read(T, R, P, W, M, hc.HC_PATH_PREFILL_UNFUSED)
    for x, y in zip(fused, unfused):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def _host(o):
    return (o[0].cpu().numpy(), o[1].cpu().numpy().view(np.uint16),
            o[2].cpu().numpy().view(np.uint16))


def test_upmix_stage_rerun_matches_the_read(weights):
    """The up + gate + mix stage run again on the read's lo gives the read's bits,
    fused and unfused; on the same lo the bf16-lo stage gives the bits of a bf16-lo
    read (every tile-path read leaves lo as its three bf16 terms, the first of which
    is lo rounded once to bf16); a stage for more tokens than the last read is
    refused."""
    w, W = weights
    T = 260
    a = synth.make_activations(14, T, True)
    R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
    ref16 = gpu_read(T, R, P, W, M, hc.HC_PATH_PREFILL_BF16_LO)
    ref = gpu_read(T, R, P, W, M, hc.HC_PATH_PREFILL)
    for path in (hc.HC_PATH_PREFILL, hc.HC_PATH_PREFILL_UNFUSED):
        o = alloc_out(T)
        hc.hc_read_upmix(path, T, R, P, W["W_up"], M, *o)
        torch.cuda.synchronize()
        for x, y in zip(ref, _host(o)):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    o = alloc_out(T)
    hc.hc_read_upmix(hc.HC_PATH_PREFILL_BF16_LO, T, R, P, W["W_up"], M, *o)
    torch.cuda.synchronize()
    for x, y in zip(ref16, _host(o)):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    with pytest.raises(hc.HcReadError):
        hc.hc_read_upmix(hc.HC_PATH_PREFILL, T + 1, R, P, W["W_up"], M, *o)
    with pytest.raises(hc.HcReadError):
        hc.hc_read_upmix(hc.HC_PATH_DECODE, T, R, P, W["W_up"], M, *o)


def _bf16_lo(T):
    lo = torch.empty((T, 320), dtype=torch.int16, device="cuda")
    hc.hc_read_lo_bf16(T, lo)
    torch.cuda.synchronize()
    return lo.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("T,with_P,seed", [(300, True, 31), (2000, True, 32), (8192, False, 100)])
def test_bf16_lo_path_against_the_read_from_its_lo(weights, T, with_P, seed):
    """The pages' prefill numerics: lo rounded once to bf16 for a one-term bf16 up
    GEMM. Its output matches, to the fp32 tolerance, the oracle's read computed from
    that same bf16 lo (exported by the library); the exported lo is the bf16
    rounding of the exact lo, within the fp32 path's own error; and the path is
    bitwise repeatable."""
    w, W = weights
    if T == 8192:
        a = synth.make_prefill_chunk(seed, T)
        a["P"] = None
    else:
        a = synth.make_activations(seed, T, with_P)
    R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
    got = gpu_read(T, R, P, W, M, hc.HC_PATH_PREFILL_BF16_LO)
    lo_bits = _bf16_lo(T)
    rng = np.random.default_rng(seed)
    idx = np.arange(T) if T <= 512 else np.unique(np.concatenate(
        [np.arange(128), np.arange(T - 128, T), rng.choice(T, 256, replace=False)]))
    Ps = None if a["P"] is None else a["P"][idx]
    lo = O.bf16_bits_to_f64(lo_bits[idx])
    want = O.hc_read_from_lo(a["R"][idx], Ps, lo, w["W_up"], a["Rmix"][idx])
    assert_matches_oracle(tuple(x[idx] for x in got), want)
    exact = O.hc_read(a["R"][idx], Ps, w["w_norm"], w["W_down"], w["W_up"], a["Rmix"][idx],
                      EPS, stages=True)["lo"]
    # half a bf16 ulp of rounding (at most 2^-8 of the value), plus the fp32 path's error
    bound = np.abs(exact) * 2.0 ** -8 + 2e-6 * np.abs(exact).max()
    assert np.all(np.abs(lo - exact) <= bound)
    again = gpu_read(T, R, P, W, M, hc.HC_PATH_PREFILL_BF16_LO)
    for x, y in zip(got, again):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    assert hc.hc_read_status() == 0


def test_prefill_bitwise_repeatable_and_pending_write(weights):
    w, W = weights
    T = 260
    a = synth.make_activations(12, T, True)
    R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
    first = gpu_read(T, R, P, W, M, hc.HC_PATH_PREFILL)
    for _ in range(3):
        again = gpu_read(T, R, P, W, M, hc.HC_PATH_PREFILL)
        for x, y in zip(first, again):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    pre = gpu_read(T, dev_f32((a["R"] + a["P"]).astype(np.float32)), None, W, M,
                   hc.HC_PATH_PREFILL)
    for x, y in zip(first, pre):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    assert hc.hc_read_status() == 0


@pytest.mark.skipif(bool(os.environ.get("HC_READ_DECODE_MAX_T")),
                    reason="the environment moves HC_PATH_AUTO's crossover")
@pytest.mark.parametrize("T,path", [(48, hc.HC_PATH_DECODE), (49, hc.HC_PATH_PREFILL)])
def test_auto_path_switches_at_48_tokens(weights, T, path):
    """HC_PATH_AUTO runs the decode kernels up to 48 tokens (the measured crossover of the
    one-pass decode and the tile path) and the tile path above: its bits are those of
    the path it picks, and both match the oracle."""
    w, W = weights
    a = synth.make_activations(60 + T, T, True)
    R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
    auto = gpu_read(T, R, P, W, M)
    forced = gpu_read(T, R, P, W, M, path)
    for x, y in zip(auto, forced):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    want = O.hc_read(a["R"], a["P"], w["w_norm"], w["W_down"], w["W_up"], a["Rmix"], EPS)
    assert_matches_oracle(auto, want)


def test_decode_and_prefill_paths_agree(weights):
    w, W = weights
    for T in (1, 5, 8):
        a = synth.make_activations(13 + T, T, True)
        R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
        d = gpu_read(T, R, P, W, M, hc.HC_PATH_DECODE)
        p = gpu_read(T, R, P, W, M, hc.HC_PATH_PREFILL)
        from _hc import rel_diff
        assert rel_diff(d[0], p[0]) <= 2 * TOL_F32


@pytest.mark.parametrize("T,with_P,seed", [(1, True, 41), (129, True, 42), (300, False, 43),
                                           (2000, True, 44), (8192, False, 101)])
def test_readout_y_against_oracle(weights, T, with_P, seed):
    """The 2560-wide read-out (y = sum of the gated streams, with its images) through
    hc_read_y, against the oracle's; long chunks on sampled tokens."""
    w, W = weights
    if T == 8192:
        a = synth.make_prefill_chunk(seed, T)
        a["P"] = None
    else:
        a = synth.make_activations(seed, T, with_P)
    R, P = dev_f32(a["R"]), dev_f32(a["P"])
    shape = (T, synth.WIDTH)
    o = (torch.empty(shape, dtype=torch.float32, device="cuda"),
         torch.empty(shape, dtype=torch.int16, device="cuda"),
         torch.empty(shape, dtype=torch.int16, device="cuda"))
    hc.hc_read_y(T, R, P, W["w_norm"], W["W_down"], W["W_up"], *o)
    torch.cuda.synchronize()
    got = _host(o)
    rng = np.random.default_rng(seed)
    idx = np.arange(T) if T <= 512 else np.unique(np.concatenate(
        [np.arange(128), np.arange(T - 128, T), rng.choice(T, 256, replace=False)]))
    Ps = None if a["P"] is None else a["P"][idx]
    want = O.hc_read_y(a["R"][idx], Ps, w["w_norm"], w["W_down"], w["W_up"], EPS)
    assert_matches_oracle(tuple(x[idx] for x in got), want)
    assert bool(torch.isfinite(o[0]).all())
    assert hc.hc_read_status() == 0


def test_back_to_back_tile_reads_do_not_see_each_others_scratch(weights):
    """Tile-path reads of alternating kinds (bf16 lo, then fp32-accurate) enqueued back
    to back with no synchronisation: each must give the bits of the same read run
    alone, so no kernel may read scratch (lo, partials) before the previous kernel
    has written it or after the next read has overwritten it."""
    w, W = weights
    T = 4096
    c = synth.make_prefill_chunk(102, T)
    R, M = dev_f32(c["R"]), dev_f32(c["Rmix"])
    ref = gpu_read(T, R, None, W, M, hc.HC_PATH_PREFILL)
    ref16 = gpu_read(T, R, None, W, M, hc.HC_PATH_PREFILL_BF16_LO)
    outs = []
    for _ in range(6):
        for path in (hc.HC_PATH_PREFILL_BF16_LO, hc.HC_PATH_PREFILL):
            o = alloc_out(T)
            hc.hc_read_path(path, T, R, None, W["w_norm"], W["W_down"], W["W_up"], M, *o)
            outs.append((path, o))
    torch.cuda.synchronize()
    for path, o in outs:
        want = ref16 if path == hc.HC_PATH_PREFILL_BF16_LO else ref
        for x, y in zip(want, _host(o)):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


@pytest.mark.parametrize("T", [3, 300])
def test_reads_captured_in_a_cuda_graph(weights, T):
    """A read captured in a CUDA graph (how a serving step calls it) and replayed gives
    the bits of the same read called directly: the launch needs no host work that a
    capture cannot hold, decode (T = 3) and tile path (T = 300) alike."""
    w, W = weights
    a = synth.make_activations(77 + T, T, True)
    R, P, M = dev_f32(a["R"]), dev_f32(a["P"]), dev_f32(a["Rmix"])
    ref = gpu_read(T, R, P, W, M)
    o = _poisoned_out(T)
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        hc.hc_read(T, R, P, W["w_norm"], W["W_down"], W["W_up"], M, *o, stream=st)
        st.synchronize()
        with torch.cuda.graph(g, stream=st):
            hc.hc_read(T, R, P, W["w_norm"], W["W_down"], W["W_up"], M, *o, stream=st)
    for _ in range(2):
        for x in o:
            x.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        for x, y in zip(ref, _host(o)):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    assert hc.hc_read_status() == 0


def _poisoned_out(T):
    """Output tensors filled with NaN / all-ones bits, so a value that no kernel wrote
    cannot pass for a correct one left over from an earlier run."""
    shape = (T, synth.N_STREAMS, synth.WIDTH)
    return (torch.full(shape, float("nan"), dtype=torch.float32, device="cuda"),
            torch.full(shape, -1, dtype=torch.int16, device="cuda"),
            torch.full(shape, -1, dtype=torch.int16, device="cuda"))


def test_up_tile_repeats_bitwise_into_poisoned_outputs(weights):
    """The up tile's epilogue groups each stream R through their own ring of slots and
    tiles are handed out at run time, so which CTA takes which tile, and how far one
    epilogue group runs ahead of the other, change from run to run. Every run of the
    up + gate + mix stage, fused and unfused, into fresh poisoned outputs must give
    the bits of the first read (a group that read a slot before its data landed
    would differ in that step's columns)."""
    w, W = weights
    T = 8192
    c = synth.make_prefill_chunk(100, T)
    R, M = dev_f32(c["R"]), dev_f32(c["Rmix"])
    o = _poisoned_out(T)
    hc.hc_read_path(hc.HC_PATH_PREFILL, T, R, None, W["w_norm"], W["W_down"], W["W_up"], M, *o)
    ref = o
    for rep in range(8):
        path = hc.HC_PATH_PREFILL_UNFUSED if rep % 2 == 0 else hc.HC_PATH_PREFILL
        o = _poisoned_out(T)
        hc.hc_read_upmix(path, T, R, None, W["W_up"], M, *o)
        for x, y in zip(ref, o):
            assert bool(torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x,
                                    y.view(torch.int32) if y.dtype == torch.float32 else y)), rep
    assert hc.hc_read_status() == 0


def test_readout_y_repeats_bitwise_into_poisoned_outputs(weights):
    """The y read-out's epilogue releases each R slot as soon as it has read it, so the
    slot's next TMA fill can land right after; four repeats of an 8,192-token read
    into fresh poisoned outputs give the same bits (a read of the slot that the next
    fill overtook would differ in that step's columns of one token)."""
    w, W = weights
    T = 8192
    c = synth.make_prefill_chunk(103, T)
    R = dev_f32(c["R"])
    shape = (T, synth.WIDTH)
    ref = None
    for rep in range(4):
        o = (torch.full(shape, float("nan"), dtype=torch.float32, device="cuda"),
             torch.full(shape, -1, dtype=torch.int16, device="cuda"),
             torch.full(shape, -1, dtype=torch.int16, device="cuda"))
        hc.hc_read_y(T, R, None, W["w_norm"], W["W_down"], W["W_up"], *o)
        if ref is None:
            ref = o
            continue
        for x, y in zip(ref, o):
            assert bool(torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x,
                                    y.view(torch.int32) if y.dtype == torch.float32 else y)), rep
    assert hc.hc_read_status() == 0


@pytest.mark.parametrize("T,path", [(3, hc.HC_PATH_DECODE), (4, hc.HC_PATH_DECODE_ONE_KERNEL),
                                    (200, hc.HC_PATH_PREFILL)])
def test_stream_permutation_equivariance(weights, T, path):
    """Relabelling the four streams consistently (residual and pending write, w_norm
    rows, W_down column blocks, W_up row blocks, the mix's rows and columns) relabels
    the output streams. The GPU sums streams in a fixed order, so the two reads agree
    to the fp32 tolerance, not bit for bit."""
    w, W = weights
    a = synth.make_activations(61 + T, T, True)
    C = synth.WIDTH
    perm = np.array([2, 0, 3, 1])
    kperm = (perm[:, None] * C + np.arange(C)[None, :]).reshape(-1)
    base = gpu_read(T, dev_f32(a["R"]), dev_f32(a["P"]), W, dev_f32(a["Rmix"]), path)
    Wp = {"w_norm": dev_u16(w["w_norm"][perm]), "W_down": dev_u16(w["W_down"][:, kperm]),
          "W_up": dev_u16(w["W_up"][kperm])}
    moved = gpu_read(T, dev_f32(a["R"][:, perm]), dev_f32(a["P"][:, perm]), Wp,
                     dev_f32(a["Rmix"][:, perm][:, :, perm]), path)
    assert rel_diff(moved[0], base[0][:, perm]) <= TOL_F32
