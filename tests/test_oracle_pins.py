"""Pins for the CPU oracle: checks against things other than the oracle itself.

* brute force in 50-digit decimal arithmetic with explicit index loops on tiny
  shapes (written from the definitions of the steps, not from the oracle's code);
* hand-worked golden cases (tests/golden/), each with its derivation and source;
* closed forms: zero up weights (gate exactly 1/2), zero norm weights, identity
  and permutation mixes, one-hot down/up weights, constant streams;
* invariants: pending write == pre-added residual, token independence, stream
  permutation equivariance, exact power-of-two scaling with eps = 0;
* textbook routines from another library: torch's ``rms_norm``, float64 matmul,
  ``sigmoid`` and ``einsum``; the converters against torch's casts (the bf16
  encoder on all 2^32 fp32 patterns, the bf16 decoder on all 2^16).

A final test plants mistakes in the oracle (transposed operands, a flipped sign,
a dropped factor, eps outside the root, the mix read the wrong way round) and
checks that the brute-force pin catches every one; another plants four in the
bf16 encoder (truncation, ties away from zero, the wrong parity bit, NaN carried
into infinity) and checks that the converter pin catches them.
"""
import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

from oracle import hc_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def bf16(x):
    """float values -> bf16 bits by torch's cast (used to build exact inputs)."""
    t = torch.tensor(np.asarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def rand_case(seed, T, n, C, r, with_P=True, dyadic=False):
    g = np.random.default_rng(seed)
    if dyadic:
        # multiples of 1/8 in [-4, 4]: every fp32 sum of two is exact
        R = (g.integers(-32, 33, (T, n, C)) / 8.0).astype(F32)
        P = (g.integers(-8, 9, (T, n, C)) / 8.0).astype(F32) if with_P else None
    else:
        R = g.standard_normal((T, n, C)).astype(F32)
        P = (0.1 * g.standard_normal((T, n, C))).astype(F32) if with_P else None
    w = bf16(1.0 + 0.1 * g.standard_normal((n, C)))
    Wd = bf16(0.3 * g.standard_normal((r, n * C)))
    Wu = bf16(0.3 * g.standard_normal((n * C, r)))
    M = g.standard_normal((T, n, n)).astype(F32)
    return R, P, w, Wd, Wu, M


# ----------------------------------------------------------------------------
# brute force, 50 significant digits, explicit loops
# ----------------------------------------------------------------------------

def _dec_bf16(bits):
    return Decimal(float(np.array(int(bits) << 16, dtype=np.uint32).view(np.float32)))


def brute_force(R, P, w, Wd, Wu, M, eps):
    """Every step by its definition, in Decimal, one index at a time.
    Returns float64 copies of rs, lo, u, gated, mixed."""
    getcontext().prec = 50
    T, n, C = R.shape
    r = Wd.shape[0]
    out = {k: [] for k in ("rs", "lo", "u", "gated", "mixed")}
    one = Decimal(1)
    for t in range(T):
        # step 1: the pending write in fp32 (one IEEE addition per element)
        Rp = [[Decimal(float(F32(R[t, s, c]) + (F32(P[t, s, c]) if P is not None else F32(0))))
               for c in range(C)] for s in range(n)]
        # step 2: per-stream RMS, eps inside the root, times w_norm
        rs = []
        for s in range(n):
            ss = sum((Rp[s][c] * Rp[s][c] for c in range(C)), Decimal(0))
            rs.append(one / (ss / C + Decimal(float(eps))).sqrt())
        xn = [Rp[k // C][k % C] * _dec_bf16(w[k // C, k % C]) * rs[k // C] for k in range(n * C)]
        # step 3: down projection, rows j, columns k = s*C + c
        lo = [sum((_dec_bf16(Wd[j, k]) * xn[k] for k in range(n * C)), Decimal(0)) for j in range(r)]
        # step 4: up projection, rows i = s*C + c, then the gate on R'
        u = [sum((_dec_bf16(Wu[i, j]) * lo[j] for j in range(r)), Decimal(0)) for i in range(n * C)]
        gated = [[Rp[s][c] / (one + (-u[s * C + c]).exp()) for c in range(C)] for s in range(n)]
        # step 5: mix, row s of the 4x4 matrix against the gated streams
        mixed = [[sum((Decimal(float(M[t, s, q])) * gated[q][c] for q in range(n)), Decimal(0))
                  for c in range(C)] for s in range(n)]
        out["rs"].append([float(x) for x in rs])
        out["lo"].append([float(x) for x in lo])
        out["u"].append([float(x) for x in u])
        out["gated"].append([[float(x) for x in row] for row in gated])
        out["mixed"].append([[float(x) for x in row] for row in mixed])
    return {k: np.array(v, dtype=np.float64) for k, v in out.items()}


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def compare_to_brute(seed, T, n, C, r, with_P, eps, dyadic):
    R, P, w, Wd, Wu, M = rand_case(seed, T, n, C, r, with_P, dyadic)
    got = O.hc_read(R, P, w, Wd, Wu, M, eps, stages=True)
    ref = brute_force(R, P, w, Wd, Wu, M, eps)
    return {k: rel_err(got[k].reshape(ref[k].shape), ref[k]) for k in ref}


@pytest.mark.parametrize("C,r", [(1, 1), (2, 1), (2, 3), (8, 3)])
@pytest.mark.parametrize("with_P", [False, True])
def test_brute_force_tiny(C, r, with_P):
    errs = compare_to_brute(11 * C + r, 2, 4, C, r, with_P, 1e-6, dyadic=False)
    for k, e in errs.items():
        assert e < 1e-13, (k, e)


def test_brute_force_dyadic_eps():
    errs = compare_to_brute(5, 3, 4, 8, 3, True, 0.25, dyadic=True)
    for k, e in errs.items():
        assert e < 1e-13, (k, e)


# ----------------------------------------------------------------------------
# hand-worked golden cases
# ----------------------------------------------------------------------------

def test_golden_hand_read():
    d = json.load(open(os.path.join(GOLDEN, "hand_read_n4_c2_r2.json")))
    R = np.array(d["R"], F32)
    st = O.hc_read(R, None, bf16(d["w_norm"]), bf16(d["W_down"]), bf16(d["W_up"]),
                   np.array(d["Rmix"], F32), d["eps"], stages=True)
    e = d["expect"]
    assert np.array_equal(st["rs"], np.array(e["rs"]))
    assert np.array_equal(st["xn"].reshape(1, -1), np.array(e["xn"]))
    assert np.array_equal(st["lo"], np.array(e["lo"]))
    assert np.array_equal(st["u"], np.array(e["u"]))
    assert np.array_equal(st["mixed"][:, :, 0], np.array(e["mixed_c0"]))

    def sig(x):
        return 1.0 / (1.0 + math.exp(-x))

    want_c1 = np.array([[eval(s, {"sig": sig}) for s in row] for row in e["mixed_c1"]])
    assert np.allclose(st["mixed"][:, :, 1], want_c1, rtol=1e-15, atol=0)
    assert np.array_equal(st["out_f32"][:, :, 0], np.array(e["mixed_c0"], F32))


def test_golden_pending_write_rounding():
    d = json.load(open(os.path.join(GOLDEN, "hand_pending_write_rounding.json")))

    def h(a):
        return np.array([[[int(x, 16) for x in c] for c in s] for s in a], np.uint32).view(F32)

    R, P, want = h(d["R_hex"]), h(d["P_hex"]), h(d["expect_Rp_hex"])
    n, C = 4, 2
    f32, _, _ = O.hc_read(R, P, bf16(np.ones((n, C))), bf16(np.ones((1, n * C))),
                          bf16(np.zeros((n * C, 1))), np.eye(n, dtype=F32)[None], 1e-6)
    assert np.array_equal(f32.view(np.uint32), (want * F32(0.5)).view(np.uint32))
    assert np.array_equal(O.pending_write(R, P).view(np.uint32), want.view(np.uint32))


# ----------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------

def test_zero_up_weights_gate_half():
    R, P, w, Wd, _, M = rand_case(1, 3, 4, 16, 5)
    Wu = bf16(np.zeros((64, 5)))
    st = O.hc_read(R, P, w, Wd, Wu, M, 1e-6, stages=True)
    Rp = (R + P).astype(np.float64)
    want = np.zeros_like(Rp)
    for t in range(3):
        for s in range(4):
            for q in range(4):
                want[t, s] += float(M[t, s, q]) * (Rp[t, q] * 0.5)
    assert np.array_equal(st["u"], np.zeros((3, 64)))
    assert np.array_equal(st["mixed"], want)


def test_zero_norm_weights():
    R, P, _, Wd, Wu, M = rand_case(2, 2, 4, 8, 3)
    st = O.hc_read(R, P, bf16(np.zeros((4, 8))), Wd, Wu, M, 1e-6, stages=True)
    assert np.array_equal(st["lo"], np.zeros((2, 3)))
    assert np.array_equal(st["gated"], (R + P).astype(np.float64) * 0.5)


def test_identity_mix_is_gated():
    R, P, w, Wd, Wu, _ = rand_case(3, 2, 4, 8, 3)
    I = np.broadcast_to(np.eye(4, dtype=F32), (2, 4, 4)).copy()
    st = O.hc_read(R, P, w, Wd, Wu, I, 1e-6, stages=True)
    assert np.array_equal(st["mixed"], st["gated"])


def test_permutation_mix_orientation():
    """Row s of Rmix selects which gated stream lands in output stream s."""
    R, P, w, Wd, Wu, _ = rand_case(4, 1, 4, 8, 3)
    perm = [2, 0, 3, 1]
    M = np.zeros((1, 4, 4), F32)
    for s, q in enumerate(perm):
        M[0, s, q] = 1.0
    st = O.hc_read(R, P, w, Wd, Wu, M, 1e-6, stages=True)
    for s, q in enumerate(perm):
        assert np.array_equal(st["mixed"][0, s], st["gated"][0, q])


def test_one_hot_weights_pick_indices():
    """W_down = a*e(j0,k0), W_up = b*e(i0,j0): only u[i0] is non-zero and it equals
    a*b*xn[k0] with xn[k0] = R'[s0][c0] * w[s0][c0] * rs[s0], k0 = s0*C + c0."""
    n, C, r = 4, 6, 3
    R, P, w, _, _, M = rand_case(6, 1, n, C, r)
    s0, c0, j0, i0 = 2, 5, 1, 1 * C + 4
    k0 = s0 * C + c0
    Wd = np.zeros((r, n * C))
    Wd[j0, k0] = 0.5
    Wu = np.zeros((n * C, r))
    Wu[i0, j0] = -3.0
    st = O.hc_read(R, P, w, bf16(Wd), bf16(Wu), M, 1e-6, stages=True)
    Rp = (R + P)[0].astype(np.float64)
    rs = 1.0 / math.sqrt(sum(float(x) ** 2 for x in Rp[s0]) / C + 1e-6)
    wk = float(np.array(int(w[s0, c0]) << 16, np.uint32).view(F32))
    want_u = -3.0 * 0.5 * (Rp[s0, c0] * wk * rs)
    u = st["u"][0]
    assert np.count_nonzero(u) == 1 and u[i0] != 0
    assert abs(u[i0] - want_u) <= 1e-14 * abs(want_u)
    lo = st["lo"][0]
    assert np.count_nonzero(lo) == 1 and lo[j0] != 0


def test_constant_stream_rs():
    n, C, r = 4, 8, 2
    R = np.zeros((1, n, C), F32)
    vals = [3.0, -0.25, 7.5, 1e-3]
    for s, a in enumerate(vals):
        R[0, s, :] = a
    eps = 1e-6
    rs = O.rms_scale(O.pending_write(R, None), eps)
    for s, a in enumerate(vals):
        want = 1.0 / math.sqrt(float(F32(a)) ** 2 + eps)
        assert abs(rs[0, s] - want) <= 1e-15 * want


# ----------------------------------------------------------------------------
# invariants
# ----------------------------------------------------------------------------

def test_pending_write_equals_preadded():
    R, P, w, Wd, Wu, M = rand_case(7, 3, 4, 16, 5)
    a = O.hc_read(R, P, w, Wd, Wu, M, 1e-6)
    b = O.hc_read((R + P).astype(F32), None, w, Wd, Wu, M, 1e-6)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_token_independence():
    R, P, w, Wd, Wu, M = rand_case(8, 6, 4, 16, 5)
    full = O.hc_read(R, P, w, Wd, Wu, M, 1e-6, stages=True)["mixed"]
    for t in (0, 3, 5):
        one = O.hc_read(R[t:t + 1], P[t:t + 1], w, Wd, Wu, M[t:t + 1], 1e-6, stages=True)["mixed"]
        assert rel_err(one[0], full[t]) < 1e-14


def test_stream_permutation_equivariance():
    n, C, r = 4, 8, 3
    R, P, w, Wd, Wu, M = rand_case(9, 2, n, C, r)
    perm = np.array([3, 1, 0, 2])
    kperm = (perm[:, None] * C + np.arange(C)[None, :]).reshape(-1)
    base = O.hc_read(R, P, w, Wd, Wu, M, 1e-6, stages=True)["mixed"]
    moved = O.hc_read(R[:, perm], P[:, perm], w[perm], Wd[:, kperm], Wu[kperm],
                      M[:, perm][:, :, perm], 1e-6, stages=True)["mixed"]
    assert rel_err(moved, base[:, perm]) < 1e-14


def test_power_of_two_scaling_exact():
    """With eps = 0, R -> 4R and P -> 4P leave xn, lo and u unchanged and scale the
    output by exactly 4 (power-of-two scalings are exact in binary)."""
    R, P, w, Wd, Wu, M = rand_case(10, 2, 4, 16, 5)
    a = O.hc_read(R, P, w, Wd, Wu, M, 0.0, stages=True)
    b = O.hc_read(R * F32(4), P * F32(4), w, Wd, Wu, M, 0.0, stages=True)
    assert np.array_equal(a["xn"], b["xn"])
    assert np.array_equal(a["u"], b["u"])
    assert np.array_equal(b["out_f32"], a["out_f32"] * F32(4))


# ----------------------------------------------------------------------------
# textbook routines from another library
# ----------------------------------------------------------------------------

def test_steps_against_torch():
    n, C, r = 4, 64, 16
    R, P, w, Wd, Wu, M = rand_case(12, 5, n, C, r)
    eps = 1e-6
    st = O.hc_read(R, P, w, Wd, Wu, M, eps, stages=True)
    Rp = torch.from_numpy((R + P).astype(np.float64))
    w64 = torch.from_numpy(w.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64)
    xn = torch.stack([torch.nn.functional.rms_norm(Rp[:, s], (C,), weight=w64[s], eps=eps)
                      for s in range(n)], dim=1)
    assert rel_err(st["xn"], xn.numpy()) < 1e-14
    Wd64 = torch.from_numpy(Wd.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64)
    Wu64 = torch.from_numpy(Wu.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64)
    lo = torch.matmul(xn.reshape(5, -1), Wd64.t())
    assert rel_err(st["lo"], lo.numpy()) < 1e-13
    u = torch.matmul(lo, Wu64.t())
    assert rel_err(st["u"], u.numpy()) < 1e-13
    gated = Rp * torch.sigmoid(u.reshape(5, n, C))
    assert rel_err(st["gated"], gated.numpy()) < 1e-13
    mixed = torch.einsum("tsq,tqc->tsc", torch.from_numpy(M.astype(np.float64)), gated)
    assert rel_err(st["mixed"], mixed.numpy()) < 1e-13
    assert np.array_equal(st["out_f32"], mixed.to(torch.float32).numpy())


# ----------------------------------------------------------------------------
# converters
# ----------------------------------------------------------------------------

def _stratified_f32_bits():
    """Every high half-word (sign, exponent, top 7 mantissa bits) with the low
    half-words that decide rounding: 0, 1, just below / at / above the bf16
    midpoint, all ones, plus random ones."""
    hi = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = [0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x1000, 0x0FFF, 0x2000, 0xE000]
    rng = np.random.default_rng(0)
    lows += [int(x) for x in rng.integers(0, 1 << 16, 6)]
    return np.concatenate([hi | np.uint32(lo) for lo in lows])


def _bf16_encoder_mismatches(encode) -> int:
    """Stratified fp32 patterns on which ``encode`` differs from torch's cast
    (NaN inputs must give a NaN)."""
    bits = _stratified_f32_bits()
    x = bits.view(F32)
    mine = encode(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    bad = int(np.count_nonzero(mine[~nan] != ref[~nan]))
    with np.errstate(invalid="ignore"):
        bad += int(np.count_nonzero(~np.isnan(O.bf16_bits_to_f64(mine[nan]))))
    return bad


def test_bf16_encoder_against_torch():
    assert _bf16_encoder_mismatches(O.f32_to_bf16_bits) == 0


def _bf16_encoder_mutants():
    def u32(x):
        return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)

    def truncate(x):             # no rounding at all
        return (u32(x) >> np.uint64(16)).astype(np.uint16)

    def ties_away(x):            # half-way cases rounded away from zero
        return ((u32(x) + np.uint64(0x8000)) >> np.uint64(16)).astype(np.uint16)

    def ties_odd_lsb(x):         # the kept bit's parity read from the wrong place
        u = u32(x)
        return ((u + np.uint64(0x7FFF) + ((u >> np.uint64(15)) & np.uint64(1))) >> np.uint64(16)).astype(np.uint16)

    def nan_to_inf(x):           # rounding carries a NaN with a low payload into infinity
        u = u32(x)
        return ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)).astype(np.uint16)

    return {"truncate": truncate, "ties_away": ties_away, "ties_odd_lsb": ties_odd_lsb,
            "nan_to_inf": nan_to_inf}


@pytest.mark.parametrize("name", list(_bf16_encoder_mutants().keys()))
def test_bf16_encoder_mistakes_are_caught(name):
    """The converter pin fails on plausible encoder mistakes."""
    assert _bf16_encoder_mismatches(_bf16_encoder_mutants()[name]) > 0


def test_bf16_encoder_exhaustive():
    """All 2^32 fp32 bit patterns through the oracle's bf16 encoder, against
    torch's cast, in blocks of 2^24 over a spawn pool (about half a minute on
    eight cores)."""
    import multiprocessing as mp

    import _converter_sweep as S

    blocks = range(1 << (32 - S.BLOCK_BITS))
    workers = max(1, min(16, os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(workers) as pool:
        results = pool.map(S.check_block, blocks, chunksize=1)
    bad = [(k, n, hex(first)) for k, n, first in results if n]
    assert len(results) == len(blocks) and not bad, bad[:4]


def test_bf16_decoder_exhaustive():
    """All 2^16 bf16 bit patterns through the oracle's decoder, against torch's
    bfloat16 -> float64 cast (NaNs compared as NaNs)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):   # signalling NaNs quieted by the widening
        mine = O.bf16_bits_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))


def test_fp16_encoder_against_torch():
    bits = _stratified_f32_bits()
    # fp16 rounding is decided 13 bits down: add patterns around that midpoint
    extra = (np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)) | np.uint32(0x1000)
    extra2 = (np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)) | np.uint32(0x0FFF)
    x = np.concatenate([bits, extra, extra2]).view(F32)
    mine = O.f32_to_f16_bits(x)
    ref = torch.from_numpy(x.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_converters_hand_values():
    enc_b = lambda v: int(O.f32_to_bf16_bits(np.array([v], F32))[0])
    enc_h = lambda v: int(O.f32_to_f16_bits(np.array([v], F32))[0])
    f = lambda b: np.array([b], np.uint32).view(F32)[0]
    assert enc_b(1.0) == 0x3F80 and enc_b(-2.0) == 0xC000
    assert enc_b(f(0x3F808000)) == 0x3F80      # 1 + 2^-8: tie, even neighbour 1
    assert enc_b(f(0x3F818000)) == 0x3F82      # 1 + 3*2^-8: tie, even neighbour up
    assert enc_b(f(0x3F808001)) == 0x3F81      # just above the tie
    assert enc_b(f(0x7F7FFFFF)) == 0x7F80      # FLT_MAX rounds to infinity
    assert enc_b(f(0x00000001)) == 0x0000      # smallest fp32 subnormal
    assert enc_h(65504.0) == 0x7BFF and enc_h(65520.0) == 0x7C00
    assert enc_h(f(0x477FEFFF)) == 0x7BFF      # just below the overflow tie
    assert enc_h(2.0 ** -24) == 0x0001 and enc_h(2.0 ** -25) == 0x0000
    assert enc_h(1.5 * 2.0 ** -24) == 0x0002   # tie between subnormals 1 and 2
    assert O.bf16_bits_to_f64(np.array([0x0001], np.uint16))[0] == 2.0 ** -133
    assert O.bf16_bits_to_f64(np.array([0x7F80], np.uint16))[0] == np.inf


# ----------------------------------------------------------------------------
# planted mistakes must be caught
# ----------------------------------------------------------------------------

def _mutants():
    F64 = np.float64

    def down_T(xn, Wb):          # reads W_down as [in][out]
        Wd = O.bf16_bits_to_f64(Wb)
        x = xn.reshape(xn.shape[0], -1)
        return x @ Wd.reshape(-1, Wd.shape[0])

    def mix_T(g, M):             # mix read with the matrix transposed
        M = np.asarray(M, F64)
        return np.einsum("tqs,tqc->tsc", M, g)

    def gate_no_R(u, Rp):        # gate without the residual
        T, n, C = Rp.shape
        return 1.0 / (1.0 + np.exp(-u.reshape(T, n, C)))

    def gate_sign(u, Rp):        # sigmoid of -u
        T, n, C = Rp.shape
        return Rp.astype(F64) / (1.0 + np.exp(u.reshape(T, n, C)))

    def rs_sum(Rp, eps):         # sum instead of mean
        x = Rp.astype(F64)
        return 1.0 / np.sqrt(np.sum(x * x, axis=-1) + eps)

    def rs_eps_out(Rp, eps):     # eps outside the root
        x = Rp.astype(F64)
        return 1.0 / (np.sqrt(np.mean(x * x, axis=-1)) + eps)

    def norm_no_w(Rp, w, rs):    # w_norm dropped
        return Rp.astype(F64) * rs[:, :, None]

    def pw_dropped(R, P):        # pending write ignored
        return np.asarray(R, np.float32).copy()

    def up_stream_major(lo, Wb): # W_up rows taken as c*n + s
        Wu = O.bf16_bits_to_f64(Wb)
        n4C = Wu.shape[0]
        C = n4C // 4
        idx = (np.arange(4)[:, None] + 4 * np.arange(C)[None, :]).reshape(-1)
        return lo @ Wu[idx].T

    return {
        "down": down_T, "mix": mix_T, "gate": gate_no_R, "gate ": gate_sign,
        "rms_scale": rs_sum, "rms_scale ": rs_eps_out, "normalise": norm_no_w,
        "pending_write": pw_dropped, "up": up_stream_major,
    }


@pytest.mark.parametrize("name", list(_mutants().keys()))
def test_planted_mistakes_are_caught(name, monkeypatch):
    fn = _mutants()[name]
    monkeypatch.setattr(O, name.strip(), fn)
    errs = compare_to_brute(3, 2, 4, 8, 3, True, 0.5, dyadic=False)
    assert max(errs.values()) > 1e-6, (name, errs)


def test_read_from_lo_is_the_read_after_its_down_projection():
    """hc_read_from_lo on the exact lo reproduces the whole read bit for bit (same
    float64 steps); on a different lo it differs, so lo is really its input."""
    rng = np.random.default_rng(77)
    T, n, C, r = 3, 4, 16, 5
    R = rng.standard_normal((T, n, C)).astype(np.float32)
    P = (0.1 * rng.standard_normal((T, n, C))).astype(np.float32)
    w_norm = O.f32_to_bf16_bits((1 + 0.1 * rng.standard_normal((n, C))).astype(np.float32))
    W_down = O.f32_to_bf16_bits((0.2 * rng.standard_normal((r, n * C))).astype(np.float32))
    W_up = O.f32_to_bf16_bits((0.2 * rng.standard_normal((n * C, r))).astype(np.float32))
    logits = rng.standard_normal((T, n, n))
    Rmix = (np.exp(logits) / np.exp(logits).sum(-1, keepdims=True)).astype(np.float32)
    st = O.hc_read(R, P, w_norm, W_down, W_up, Rmix, 1e-6, stages=True)
    got = O.hc_read_from_lo(R, P, st["lo"], W_up, Rmix)
    for x, y in zip(got, (st["out_f32"], st["out_bf16"], st["out_fp16"])):
        assert np.array_equal(x, y)
    other = O.hc_read_from_lo(R, P, st["lo"] * 1.5, W_up, Rmix)
    assert not np.array_equal(other[0], st["out_f32"])


def test_readout_y_is_the_mix_with_a_row_of_ones():
    """y = sum of the gated streams equals output stream 0 of the read whose mix
    matrix has an all-ones first row (the mix is pinned by brute force and by the
    permutation test), bit for bit: multiplying by 1 is exact and both sum q = 0..3
    in order."""
    rng = np.random.default_rng(78)
    T, n, C, r = 3, 4, 16, 5
    R = rng.standard_normal((T, n, C)).astype(np.float32)
    P = (0.1 * rng.standard_normal((T, n, C))).astype(np.float32)
    w_norm = O.f32_to_bf16_bits((1 + 0.1 * rng.standard_normal((n, C))).astype(np.float32))
    W_down = O.f32_to_bf16_bits((0.2 * rng.standard_normal((r, n * C))).astype(np.float32))
    W_up = O.f32_to_bf16_bits((0.2 * rng.standard_normal((n * C, r))).astype(np.float32))
    ones = np.ones((T, n, n), dtype=np.float32)
    full = O.hc_read(R, P, w_norm, W_down, W_up, ones, 1e-6)
    y = O.hc_read_y(R, P, w_norm, W_down, W_up, 1e-6)
    for a, b in zip(y, full):
        assert np.array_equal(a, b[:, 0, :])
    # and it is the plain sum of the gated streams of the staged read
    st = O.hc_read(R, P, w_norm, W_down, W_up, ones, 1e-6, stages=True)
    assert np.allclose(O.readout_y(st["gated"]), st["gated"].sum(axis=1), rtol=1e-15, atol=0)


def test_read_tokens_is_the_read_of_those_rows():
    """hc_read_tokens (the checker of long chunks on sampled tokens) returns rows
    ``idx`` of the whole read, for unsorted and repeated indices, with and without
    the pending write: within float64 rounding of the batched matrix products, and
    bitwise for the images wherever the fp32 values agree bitwise."""
    rng = np.random.default_rng(79)
    T, n, C, r = 9, 4, 16, 5
    R = rng.standard_normal((T, n, C)).astype(np.float32)
    P = (0.1 * rng.standard_normal((T, n, C))).astype(np.float32)
    w_norm = O.f32_to_bf16_bits((1 + 0.1 * rng.standard_normal((n, C))).astype(np.float32))
    W_down = O.f32_to_bf16_bits((0.2 * rng.standard_normal((r, n * C))).astype(np.float32))
    W_up = O.f32_to_bf16_bits((0.2 * rng.standard_normal((n * C, r))).astype(np.float32))
    logits = rng.standard_normal((T, n, n))
    Rmix = (np.exp(logits) / np.exp(logits).sum(-1, keepdims=True)).astype(np.float32)
    idx = np.array([7, 0, 3, 3, 8])
    for Pv in (P, None):
        full = O.hc_read(R, Pv, w_norm, W_down, W_up, Rmix, 1e-6)
        some = O.hc_read_tokens(idx, R, Pv, w_norm, W_down, W_up, Rmix, 1e-6)
        assert some[0].shape == (len(idx), n, C)
        np.testing.assert_allclose(some[0], full[0][idx], rtol=1e-6, atol=1e-7)
        same = some[0] == full[0][idx]
        assert same.mean() > 0.99
        for k in (1, 2):
            assert np.array_equal(some[k][same], full[k][idx][same])
    # a token's row does not depend on which other tokens are read with it: a wrong
    # index (off by one) shows up
    shifted = O.hc_read_tokens(idx + 1 - (idx == 8) * 9, R, P, w_norm, W_down, W_up, Rmix, 1e-6)
    assert not np.allclose(shifted[0], O.hc_read(R, P, w_norm, W_down, W_up, Rmix, 1e-6)[0][idx])
