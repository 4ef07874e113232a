"""The algorithmic byte counts behind every roofline fraction the bench reports.

Each count is what the read must move at the least: every weight read once, every
activation read once, every output written once, nothing else. The figures below
are worked out by hand from the shapes (4 streams x 2560 columns, rank 320, bf16
weights, fp32 activations, a 4x4 fp32 mix per token, outputs in fp32 + bf16 + fp16).
"""
import bench

W_DOWN = 320 * 10240 * 2          # 6,553,600 B of bf16
W_UP = 10240 * 320 * 2            # 6,553,600 B
W_NORM = 4 * 2560 * 2             # 20,480 B
R_TOKEN = 4 * 2560 * 4            # 40,960 B of fp32 residual (P has the same size)
MIX_TOKEN = 16 * 4                # 64 B
OUT_TOKEN = 4 * 2560 * (4 + 2 + 2)   # 81,920 B: fp32 plus the two 16-bit images
LO_TOKEN = 320 * 4                # 1,280 B of fp32 lo


def test_decode_read_bytes():
    assert bench.WEIGHT_BYTES == W_DOWN + W_UP + W_NORM == 13_127_680
    assert bench.read_bytes(1, False) == 13_250_624
    assert bench.read_bytes(4, True) == 13_783_296
    assert bench.read_bytes(8, True) == 14_438_912
    for T in (1, 3, 8):
        for p in (False, True):
            per = R_TOKEN * (2 if p else 1) + MIX_TOKEN + OUT_TOKEN
            assert bench.read_bytes(T, p) == W_DOWN + W_UP + W_NORM + T * per


def test_decode_floors_at_the_measured_copy_rate():
    """The 4-token read with a pending write at 6,792.7 GB/s: about 2.03 us."""
    us = bench.read_bytes(4, True) / 6792.7e9 * 1e6
    assert 2.02 < us < 2.04


def test_prefill_byte_counts():
    assert bench.prefill_upmix_bytes(8192) == W_UP + 8192 * (LO_TOKEN + R_TOKEN + MIX_TOKEN + OUT_TOKEN)
    assert bench.prefill_upmix_bytes(8192) == 1_024_196_608
    assert bench.prefill_upmix_bytes(32768) == 4_077_125_632
    assert bench.prefill_read_bytes(8192) == W_DOWN + W_UP + W_NORM + 8192 * (R_TOKEN + MIX_TOKEN + OUT_TOKEN)


def test_sweep_is_the_verify_window():
    """Sixteen reads per step: T = 1..8, each with and without the pending write."""
    assert sorted(bench.SWEEP) == sorted((T, p) for T in range(1, 9) for p in (False, True))
    assert len(bench.SWEEP) == 16


def test_prefill_cpu_baseline_worker_times_the_oracle_read():
    """The worker the prefill CPU baseline runs in each spawned process times exactly
    the oracle read of its tokens (here two, with the bench's weights)."""
    import numpy as np
    from hyper_connection_residual_read_gb300 import synth
    from oracle.timing import timed_read
    w = synth.make_weights(0)
    c = synth.make_prefill_chunk(100, 2)
    t = timed_read((c["R"], c["Rmix"], w, float(np.float32(1e-6))))
    assert isinstance(t, float) and t > 0.0
