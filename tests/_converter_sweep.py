"""Worker for the exhaustive check of the oracle's fp32 -> bf16 encoder.

It lives in its own module so that a ``spawn`` process pool can import it by
name. Each call checks one block of 2^24 consecutive fp32 bit patterns against
torch's float32 -> bfloat16 cast (round to nearest even). The oracle's
encoder must give the same bits for every non-NaN input and a NaN for every NaN.
"""
import numpy as np

BLOCK_BITS = 24


def check_block(k: int):
    """Return (block, mismatches, first mismatching fp32 bit pattern or -1)."""
    import torch

    torch.set_num_threads(1)
    from oracle import hc_oracle as O

    lo = k << BLOCK_BITS
    bits = np.arange(lo, lo + (1 << BLOCK_BITS), dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    mine = O.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    bad = (mine != ref) & ~nan
    # a NaN input must stay a NaN: exponent all ones and a nonzero mantissa
    bad |= nan & ~(((mine & 0x7F80) == 0x7F80) & ((mine & 0x007F) != 0))
    n = int(np.count_nonzero(bad))
    first = int(bits[np.argmax(bad)]) if n else -1
    return k, n, first
