"""Seeded synthetic inputs for the hyper-connection read.

This module only draws random numbers and packs them into the storage formats of
the read's arguments. It holds none of the read's arithmetic, and both the CUDA
path and the CPU oracle are fed from it.

Recipe (one PCG64 stream per seed, values drawn as float64):

* residual ``R[T][n][C]`` fp32 ~ N(0, 1)
* pending write ``P[T][n][C]`` fp32 ~ N(0, 0.1) (standard deviation 0.1)
* ``w_norm[n][C]`` bf16 ~ 1 + N(0, 0.1)
* ``W_down[r][n*C]`` and ``W_up[n*C][r]`` bf16 ~ N(0, 0.02)
* ``Rmix[T][n][n]`` fp32: each row is the softmax (computed in float64) of
  N(0, 1) logits, so every output stream is a convex mix of the input streams.

float64 -> fp32 is round-to-nearest; bf16 is the round-to-nearest-even image of
that fp32 value, produced by torch's cast and stored as raw ``uint16`` bits.
Weight sets and activations come from separate seeds, so one weight set can be
paired with many activation seeds. Long prefill chunks draw ``R`` directly as
float32 normals (numpy's float32 sampler), in slabs, to keep host memory and time
in proportion to the chunk.
"""
from __future__ import annotations

import numpy as np
import torch

N_STREAMS = 4
WIDTH = 2560
RANK = 320


def _to_bf16_bits(x64: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x64, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def make_weights(seed: int, n: int = N_STREAMS, C: int = WIDTH, r: int = RANK) -> dict:
    """One layer's read weights: ``w_norm``, ``W_down`` and ``W_up`` as bf16 bits."""
    g = np.random.default_rng(seed)
    w_norm = 1.0 + 0.1 * g.standard_normal((n, C))
    W_down = 0.02 * g.standard_normal((r, n * C))
    W_up = 0.02 * g.standard_normal((n * C, r))
    return {
        "w_norm": _to_bf16_bits(w_norm),
        "W_down": _to_bf16_bits(W_down),
        "W_up": _to_bf16_bits(W_up),
    }


def make_activations(seed: int, T: int, with_P: bool, n: int = N_STREAMS,
                     C: int = WIDTH) -> dict:
    """Per-token inputs: residual ``R``, optional pending write ``P``, mix ``Rmix``."""
    g = np.random.default_rng(seed)
    R = g.standard_normal((T, n, C)).astype(np.float32)
    P = (0.1 * g.standard_normal((T, n, C))).astype(np.float32) if with_P else None
    logits = g.standard_normal((T, n, n))
    e = np.exp(logits - logits.max(axis=-1, keepdims=True))
    Rmix = (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)
    return {"R": R, "P": P, "Rmix": Rmix}


def make_prefill_chunk(seed: int, T: int, n: int = N_STREAMS, C: int = WIDTH) -> dict:
    """A long chunk of tokens without a pending write, drawn in slabs of 4096 tokens
    so that peak host memory stays near the size of the result."""
    g = np.random.default_rng(seed)
    R = np.empty((T, n, C), dtype=np.float32)
    step = 4096
    for t0 in range(0, T, step):
        t1 = min(T, t0 + step)
        R[t0:t1] = g.standard_normal((t1 - t0, n, C), dtype=np.float32)
    logits = g.standard_normal((T, n, n))
    e = np.exp(logits - logits.max(axis=-1, keepdims=True))
    Rmix = (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)
    return {"R": R, "P": None, "Rmix": Rmix}
