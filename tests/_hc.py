"""Helpers shared by the GPU tests: device copies of seeded inputs, one read
through the C ABI, and the comparisons with the oracle's outputs."""
from __future__ import annotations

import numpy as np
import torch

import hyper_connection_residual_read_gb300 as hc
from hyper_connection_residual_read_gb300 import synth

# spec tolerance for fp32 `mixed`: max |gpu - oracle| / max |oracle|
TOL_F32 = 2e-6
EPS = float(np.float32(1e-6))   # the fp32 eps the library uses by default
MAX_TOKENS = 32768


def dev_u16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def dev_f32(a: np.ndarray | None) -> torch.Tensor | None:
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def dev_weights(w: dict) -> dict:
    return {k: dev_u16(v) for k, v in w.items()}


def alloc_out(T: int) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    shape = (T, synth.N_STREAMS, synth.WIDTH)
    return (torch.empty(shape, dtype=torch.float32, device="cuda"),
            torch.empty(shape, dtype=torch.int16, device="cuda"),
            torch.empty(shape, dtype=torch.int16, device="cuda"))


def gpu_read(T, R, P, W, Rmix, path=None, out=None):
    """One read through the C ABI; returns host copies (f32, bf16 bits, fp16 bits)."""
    o = out if out is not None else alloc_out(T)
    if path is None:
        hc.hc_read(T, R, P, W["w_norm"], W["W_down"], W["W_up"], Rmix, *o)
    else:
        hc.hc_read_path(path, T, R, P, W["w_norm"], W["W_down"], W["W_up"], Rmix, *o)
    torch.cuda.synchronize()
    return (o[0].cpu().numpy(), o[1].cpu().numpy().view(np.uint16),
            o[2].cpu().numpy().view(np.uint16))


def ordered16(bits: np.ndarray) -> np.ndarray:
    """Sign-magnitude 16-bit patterns -> integers in value order (+0 == -0)."""
    b = bits.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def rel_diff(got: np.ndarray, want: np.ndarray) -> float:
    d = np.max(np.abs(got.astype(np.float64) - want.astype(np.float64)))
    m = np.max(np.abs(want.astype(np.float64)))
    return float(d / m) if m > 0 else float(d)


def _decode16(bits: np.ndarray, kind: str) -> np.ndarray:
    if kind == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return bits.view(np.float16).astype(np.float64)


def _ulp16(v: np.ndarray, kind: str) -> np.ndarray:
    """Spacing of the 16-bit format at |v| (normal or subnormal)."""
    mant, emin = (7, -126) if kind == "bf16" else (10, -14)
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.exp2(e - mant)


def assert_images_close(img: np.ndarray, want_img: np.ndarray, want_f32: np.ndarray,
                        kind: str, delta: float):
    """The image is within 1 ulp of the oracle's image, or, for elements so close to
    zero that the fp32 tolerance band spans several of their ulps, within that band
    plus half an ulp of the oracle's fp32 value. Returns the fraction of elements
    that equal the oracle's image exactly."""
    d = np.abs(ordered16(img) - ordered16(want_img))
    v = _decode16(img, kind)
    band = np.abs(v - want_f32.astype(np.float64)) <= 0.5 * _ulp16(v, kind) + delta
    bad = ~((d <= 1) | band)
    assert not bad.any(), (f"{kind} image: {int(bad.sum())} elements off, e.g. "
                           f"{img[bad][:4]} vs {want_img[bad][:4]}")
    return float(np.mean(d == 0))


def assert_matches_oracle(got, want, tol=TOL_F32):
    """fp32 within max|diff|/max|value| <= tol; the images within 1 ulp of the
    oracle's images (see assert_images_close for elements near zero); and the GPU's
    own images are exactly the RNE images of its fp32 output."""
    from oracle import hc_oracle as O
    f32, b16, h16 = got
    wf, wb, wh = want
    assert np.all(np.isfinite(f32))
    r = rel_diff(f32, wf)
    assert r <= tol, f"max|diff|/max|value| = {r:.3g} > {tol}"
    delta = tol * float(np.max(np.abs(wf.astype(np.float64))))
    eq_b = assert_images_close(b16, wb, wf, "bf16", delta)
    eq_h = assert_images_close(h16, wh, wf, "fp16", delta)
    # a wrong rounding mode or a wrong element would show as far more mismatches; the
    # fp16 floor sits lower because its 11 bits resolve the fp32 error on more elements
    assert eq_b > 0.995 and eq_h > 0.99, (eq_b, eq_h)
    assert np.array_equal(b16, O.f32_to_bf16_bits(f32))
    assert np.array_equal(h16, O.f32_to_f16_bits(f32))
    return r
