"""The bench's roofline arithmetic on CPU: the algorithmic byte and FLOP counts it divides
by, checked against counts written out by hand from the definition of what a launch
must read and write."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_algorithmic_bytes_of_the_fractus1b_block():
    """Per group at C = 128, D = 64, bf16: the forward reads q, k, v (3 x 16 KB), writes o
    (16 KB) and reads and writes the fp32 carry (2 x (16 KB + 256 B)): 98,816 B.  The
    backward reads q, k, v, dO (4 x 16 KB) and S0, z0, dS_out, dz_out, and writes dq, dk,
    dv and dS0, dz0: 164,608 B."""
    tile = 128 * 64 * 2
    carry = 64 * 64 * 4 + 64 * 4
    fwd, bwd = bench.algorithmic_bytes(160, 128, 64, 2)
    assert fwd == 160 * (4 * tile + 2 * carry) == 160 * 98_816 == 15_810_560
    assert bwd == 160 * (7 * tile + 3 * carry) == 160 * 164_608 == 26_337_280


def test_threaded_long_stream_counts_every_carry_round_trip():
    """64 launches of 128 tokens move the carry in and out 64 times: 64 x the one-chunk
    forward bytes, against the single launch over 8192 tokens that moves it once."""
    one = bench.algorithmic_bytes(160, 128, 64, 2)[0]
    whole = bench.algorithmic_bytes(160, 8192, 64, 2)[0]
    carry = 160 * 2 * (64 * 64 + 64) * 4
    assert 64 * one - whole == 63 * carry
    assert bench.THREAD_CHUNK == 128


def test_cumsum_flop_model():
    """Each token updates the D x D state and reads it out once per sweep (2 D^2 FMA,
    4 D^2 FLOP); the forward makes one sweep, the backward four."""
    fwd, bwd = bench.cumsum_flop(160, 128, 64)
    assert fwd == 160 * 128 * 4 * 64 * 64
    assert bwd == 4 * fwd


def test_nominal_and_fallback_peaks():
    assert bench.NOMINAL_HBM_GBS == 7900.0
    assert bench.FALLBACK_HBM_GBS == 6800.0
