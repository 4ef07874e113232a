"""Oracle for the hyper-connection read: plain, slow, float64, on the CPU.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or runs
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may. It shares no
code with the CUDA library (its own bf16 decoder and encoder, its own step
functions) and takes every input as a plain array.

Sources (pages by title; "section" is the heading on the page):

* [UPMIX]   "#1370 prefill: opt-in STRATA_HC_UPMIX=1 on CUDA - the hyper-connection
            up projection with gr_mix_r as its epilogue (sm_80+)", sections "Why"
            and "What it does".
* [SPLIT]   "#315 hc: the multi-token hyper-connection read split finer",
            sections "What changes" and "Exactness".
* [A770]    "#2488 sycl/A770: faster hyper-connection read on Arc A-series",
            section "Summary", changes 1, 4 and 5.
* [SM75]    "#2070 sm_75: a hyper-connection up kernel for 3+ tokens and the staged
            down kernel in token pairs (bitwise)", change 1.

The pages describe kernels, never the formulas. The steps below take the plainest
reading that the pages support; every point they leave open is one of these
readings:

1. the gate is the logistic sigmoid of the up projection and it scales the
   pending-updated residual: ``gated = sigmoid(u) * R'`` (the mix "reads gated
   back with R", [UPMIX] "Why"; the epilogue prefetches "R rows", [UPMIX] "What
   it does");
2. output stream ``s`` is row ``s`` of the per-token 4x4 mix times the gated
   streams, ``mixed[s][c] = sum_q Rmix[s][q] * gated[q][c]``;
3. the RMS norm is per (token, stream) over the stream's ``C`` values, with eps
   inside the square root, scaled elementwise by ``w_norm[s][c]`` ([SPLIT] "What
   changes", norm v2/v3; [A770] change 4, "each stream's rs");
4. the flattened index of the 10240-wide axis is ``k = s*C + c`` for both the
   columns of ``W_down`` and the rows of ``W_up``; both matrices are stored
   row-major as [out][in];
5. the pending write is one fp32 addition ``R' = fl32(R + P)``; ``R`` itself is
   not written back;
6. ``lo`` (the down output) and ``xn`` (the normalised input) are exact real
   numbers here, not rounded to bf16;
7. the bf16 and fp16 images are the round-to-nearest-even images of the fp32
   ``mixed`` value (fp16 with gradual underflow, overflow to infinity).

Parity pins (tests/test_oracle_pins.py): exact brute force on tiny shapes in
50-digit decimal arithmetic, hand-derived golden cases, closed forms (zero up
weights, identity and permutation mixes, one-hot weights, constant streams),
invariants (pending write, token independence, stream permutation, power-of-two
scaling), RMS norm against torch's ``rms_norm``, the projections against torch's
float64 matmul, and the converters against torch's casts. Every function below is
covered by at least one of them.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


# ----------------------------------------------------------------------------
# storage formats
# ----------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bits -> exact float64 value (a bf16 is the top half of an fp32)."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(F64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest, ties to even; NaN stays NaN (quiet).

    Adding 0x7FFF plus the lowest kept bit and truncating rounds half-way cases to
    the even neighbour and carries into the exponent (up to infinity) as IEEE
    rounding does.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = (u + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)
    is_nan = (u & np.uint64(0x7FFFFFFF)) > np.uint64(0x7F800000)
    quiet = (u >> np.uint64(16)) | np.uint64(0x0040)
    return np.where(is_nan, quiet, rounded).astype(np.uint16)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> IEEE binary16 bits, round to nearest even, subnormals kept,
    overflow to infinity (numpy's float32 -> float16 conversion)."""
    with np.errstate(over="ignore", invalid="ignore"):
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


# ----------------------------------------------------------------------------
# the five steps, for a batch of independent tokens
# ----------------------------------------------------------------------------

def pending_write(R: np.ndarray, P: np.ndarray | None) -> np.ndarray:
    """Step 1: ``R' = fl32(R + P)`` (reading 5), or ``R`` when there is no write.
    [A770] change 4 ("the pending-updated residual"); [SPLIT] "Exactness"
    (reads run with and without the pending write)."""
    R = np.asarray(R, dtype=np.float32)
    if P is None:
        return R.copy()
    return R + np.asarray(P, dtype=np.float32)  # one IEEE fp32 addition


def rms_scale(Rp: np.ndarray, eps: float) -> np.ndarray:
    """Step 2a: ``rs[t][s] = 1 / sqrt(mean_c R'[t][s][c]^2 + eps)`` (reading 3).
    [SPLIT] "What changes" (a sum of squares and an ``rs`` per token and stream)."""
    x = Rp.astype(F64)
    C = x.shape[-1]
    ss = np.sum(x * x, axis=-1)
    return 1.0 / np.sqrt(ss / C + F64(eps))


def normalise(Rp: np.ndarray, w_norm_bits: np.ndarray, rs: np.ndarray) -> np.ndarray:
    """Step 2b: ``xn[t][s][c] = R'[t][s][c] * w_norm[s][c] * rs[t][s]``, exact.
    [SPLIT] "What changes" ("R' * w_norm ... scaled"); [A770] change 4."""
    w = bf16_bits_to_f64(w_norm_bits)
    return Rp.astype(F64) * w[None, :, :] * rs[:, :, None]


def down(xn: np.ndarray, W_down_bits: np.ndarray) -> np.ndarray:
    """Step 3: ``lo[t][j] = sum_k W_down[j][k] * xn[t][k]`` with ``k = s*C + c``
    (reading 4). [SPLIT] "What changes" (the down projection's rows);
    [A770] changes 1 and 4."""
    T = xn.shape[0]
    x = xn.reshape(T, -1)
    Wd = bf16_bits_to_f64(W_down_bits)
    return x @ Wd.T


def up(lo: np.ndarray, W_up_bits: np.ndarray) -> np.ndarray:
    """Step 4a: ``u[t][i] = sum_j W_up[i][j] * lo[t][j]`` for ``i = s*C + c``.
    [UPMIX] "Why" (the up GEMM); [SM75] change 1 (rows of ``w_up``);
    [A770] change 5 (one up row per lane)."""
    Wu = bf16_bits_to_f64(W_up_bits)
    return lo @ Wu.T


def gate(u: np.ndarray, Rp: np.ndarray) -> np.ndarray:
    """Step 4b: ``gated[t][s][c] = R'[t][s][c] / (1 + exp(-u[t][s*C + c]))``
    (reading 1). [UPMIX] "Why" (the up GEMM writes ``gated``)."""
    T, n, C = Rp.shape
    with np.errstate(over="ignore"):
        g = 1.0 / (1.0 + np.exp(-u.reshape(T, n, C)))
    return Rp.astype(F64) * g


def mix(gated: np.ndarray, Rmix: np.ndarray) -> np.ndarray:
    """Step 5: ``mixed[t][s][c] = sum_{q=0..3} Rmix[t][s][q] * gated[t][q][c]``
    (reading 2). [UPMIX] "What it does" (the mix of the 4 streams)."""
    M = np.asarray(Rmix, dtype=np.float32).astype(F64)
    T, n, C = gated.shape
    out = np.zeros((T, n, C), dtype=F64)
    for s in range(n):
        for q in range(n):
            out[:, s, :] += M[:, s, q, None] * gated[:, q, :]
    return out


def readout_y(gated: np.ndarray) -> np.ndarray:
    """The 2560-wide read-out: ``y[c] = sum_q gated[q][c]``, streams in order q =
    0..3. It is the read-out under which [UPMIX] "Why" (``gr_mix_r`` moving about
    102 KB per token: gated and residual in, one fp32 + bf16 + fp16 row of width
    C out) adds up; with it the images are taken of ``y`` as of ``mixed``."""
    y = gated[:, 0, :].copy()
    for q in range(1, gated.shape[1]):
        y = y + gated[:, q, :]
    return y


def images(mixed: np.ndarray):
    """Step 5, outputs: ``mixed`` rounded once to fp32, and the bf16 and fp16
    images of that fp32 value (reading 7). [UPMIX] "What it does" ("writes
    mixed with its BF16 / FP16 images")."""
    out_f32 = mixed.astype(np.float32)
    return out_f32, f32_to_bf16_bits(out_f32), f32_to_f16_bits(out_f32)


def hc_read(R, P, w_norm, W_down, W_up, Rmix, eps: float = 1e-6, stages: bool = False):
    """The whole read for ``T`` independent tokens.

    Shapes: ``R``, ``P`` [T][n][C] fp32 (``P`` may be None); ``w_norm`` [n][C],
    ``W_down`` [r][n*C], ``W_up`` [n*C][r] as bf16 bits (uint16); ``Rmix``
    [T][n][n] fp32. ``eps`` is used as given (pass the fp32 value the GPU uses).
    Returns ``(out_f32, out_bf16_bits, out_fp16_bits)`` or, with ``stages``, a
    dict that also holds ``Rp, rs, xn, lo, u, gated, mixed``.
    """
    Rp = pending_write(R, P)
    rs = rms_scale(Rp, eps)
    xn = normalise(Rp, w_norm, rs)
    lo = down(xn, W_down)
    u = up(lo, W_up)
    g = gate(u, Rp)
    m = mix(g, Rmix)
    f32, b16, h16 = images(m)
    if not stages:
        return f32, b16, h16
    return {"Rp": Rp, "rs": rs, "xn": xn, "lo": lo, "u": u, "gated": g, "mixed": m,
            "out_f32": f32, "out_bf16": b16, "out_fp16": h16}


def hc_read_from_lo(R, P, lo, W_up, Rmix):
    """The read after its down projection, from a given ``lo`` ([T][r], real values):
    the pending write, then the up projection, gate, mix and images (steps 4-5).
    With ``lo`` the exact down output it is the whole read. Given the bf16 ``lo`` that
    a bf16-lo tile path fed to its up GEMM, it is that path's reference: [UPMIX] "What
    it does" runs the up projection as a BF16 ``mma`` whose A operand is ``lo``."""
    Rp = pending_write(R, P)
    u = up(np.asarray(lo, dtype=F64), W_up)
    return images(mix(gate(u, Rp), Rmix))


def hc_read_y(R, P, w_norm, W_down, W_up, eps: float = 1e-6):
    """The read with ``readout_y`` in place of the mix: ``(y_f32, y_bf16, y_fp16)``,
    each [T][C]."""
    Rp = pending_write(R, P)
    lo = down(normalise(Rp, w_norm, rms_scale(Rp, eps)), W_down)
    return images(readout_y(gate(up(lo, W_up), Rp)))


def hc_read_tokens(token_ids, R, P, w_norm, W_down, W_up, Rmix, eps: float = 1e-6):
    """The read for a subset of tokens of a long chunk (tokens are independent,
    so this equals rows ``token_ids`` of the whole read)."""
    idx = np.asarray(token_ids)
    Ps = None if P is None else P[idx]
    return hc_read(R[idx], Ps, w_norm, W_down, W_up, Rmix[idx], eps)
