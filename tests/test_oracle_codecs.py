"""Pins of the oracle's scalar codecs against the format definitions.

The E2M1 and E4M3 grids are checked against values fixed by the formats
themselves (OCP 8-bit / 4-bit float definitions, which the miniTE Technical
Report section 2.2 names: E2M1 elements, E4M3 block scales); rounding is
checked at every decision boundary of the grid, so a wrong grid value, a
wrong tie rule or a wrong saturation point fails here.
"""
import struct

import numpy as np
import pytest
import torch


def f32(bits):
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def bits(x):
    return struct.unpack("<I", struct.pack("<f", x))[0]


# ---- E2M1 ----------------------------------------------------------------
E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # OCP FP4 (E2M1) magnitudes


def test_e2m1_grid_values(orc):
    for c in range(8):
        assert orc.e2m1_value(c) == E2M1_GRID[c]
        v = orc.e2m1_value(c | 8)
        assert v == -E2M1_GRID[c] and np.signbit(v)


def test_e2m1_roundtrip_all_codes(orc):
    for c in range(16):
        assert orc.e2m1_encode(orc.e2m1_value(c)) == c


@pytest.mark.parametrize("mid,expect", [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4),
                                        (2.5, 4), (3.5, 6), (5.0, 6)])
def test_e2m1_exact_ties_go_to_even_code(orc, mid, expect):
    assert orc.e2m1_encode(mid) == expect
    assert orc.e2m1_encode(-mid) == expect | 8
    lo, hi = f32(bits(mid) - 1), f32(bits(mid) + 1)
    # one float below/above the midpoint goes to the nearer code
    assert orc.e2m1_value(orc.e2m1_encode(lo)) < mid
    assert orc.e2m1_value(orc.e2m1_encode(hi)) > mid


def test_e2m1_saturation_and_sign(orc):
    for q in [6.0, 6.5, 7.0, 1e6, 3.0e38]:
        assert orc.e2m1_encode(q) == 7
        assert orc.e2m1_encode(-q) == 15
    assert orc.e2m1_encode(0.0) == 0
    assert orc.e2m1_encode(-0.0) == 8
    assert orc.e2m1_encode(-1e-30) == 8
    assert orc.e2m1_encode(1e-30) == 0


def test_e2m1_transitions_are_midpoints(orc):
    """First input of each code is the midpoint to the previous code (tie to
    even), or the float just above it (tie to the odd neighbour)."""
    for c in range(1, 8):
        mid = (E2M1_GRID[c - 1] + E2M1_GRID[c]) / 2
        first = orc.lib().orc_e2m1_first_input_of_code(c)
        expect = bits(mid) if c % 2 == 0 else bits(mid) + 1
        assert first == expect, (c, hex(first), hex(expect))


# ---- E4M3 ----------------------------------------------------------------
E4M3_KNOWN = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
              0x38: 1.0, 0x3F: 1.875, 0x40: 2.0, 0x70: 128.0, 0x78: 256.0, 0x7E: 448.0}


def test_e4m3_known_values(orc):
    for c, v in E4M3_KNOWN.items():
        assert orc.e4m3_value(c) == v
        assert orc.e4m3_value(c | 0x80) == -v
    assert np.isnan(orc.e4m3_value(0x7F))
    assert np.isnan(orc.e4m3_value(0xFF))


def test_e4m3_grid_monotone_and_roundtrip(orc):
    vals = [orc.e4m3_value(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(vals, vals[1:]))
    assert len(set(vals)) == 127
    for c in range(0x7F):
        assert orc.e4m3_encode(vals[c]) == c


def test_e4m3_transitions_are_midpoints(orc):
    vals = [orc.e4m3_value(c) for c in range(0x7F)]
    for c in range(1, 0x7F):
        mid = (vals[c - 1] + vals[c]) / 2  # exact in binary32 (<= 5 bits)
        assert np.float32(mid) == mid
        first = orc.lib().orc_e4m3_first_input_of_code(c)
        expect = bits(mid) if c % 2 == 0 else bits(mid) + 1
        assert first == expect, (hex(c), hex(first), hex(expect))


def test_e4m3_subnormal_ties_and_saturation(orc):
    assert orc.e4m3_encode(2.0 ** -10) == 0x00        # tie 0 | 2^-9 -> even 0
    assert orc.e4m3_encode(1.5 * 2.0 ** -9) == 0x02   # tie 1 | 2 -> even
    assert orc.e4m3_encode(3.5 * 2.0 ** -9) == 0x04   # tie 3 | 4 -> even
    assert orc.e4m3_encode(2.0 ** -11) == 0x00
    for t in [448.0, 460.0, 464.0, 500.0, 1e10, 3e38]:
        assert orc.e4m3_encode(t) == 0x7E


def test_e4m3_encoder_monotone_on_sample(orc):
    rng = np.random.default_rng(1)
    pats = np.sort(np.concatenate([rng.integers(0, 0x7F800000, 20000),
                                   np.arange(0x3A000000, 0x3A000000 + 4096),
                                   np.arange(0x43DF0000, 0x43E10000, 7)]))
    enc = orc.lib().orc_e4m3_encode
    codes = [enc(f32(int(p))) for p in pats]
    assert all(b >= a for a, b in zip(codes, codes[1:]))


# ---- BF16 ----------------------------------------------------------------
def test_f32_to_bf16_matches_torch_cast(orc):
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(5000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 5000),
                        np.array([0.0, -0.0, 1.0, 3.4e38, -3.4e38, 1e-40, -1e-40, 2 ** -133], np.float32)])
    # values exactly halfway between BF16 neighbours, both parities
    ties = (np.arange(1000, dtype=np.uint32) << 16 | 0x8000).view(np.float32) * 1.0
    x = np.concatenate([x, ties.astype(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.f32_to_bf16_bits(x)
    assert np.array_equal(got, ref)


def test_f64_to_bf16_rounds_once(orc):
    L = orc.lib()
    # 1 + 2^-8 is the exact midpoint between 1 and 1 + 2^-7
    assert L.orc_f64_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # just above the midpoint by less than a float ulp: a float-first cast
    # would see a tie and go to 1.0; one rounding goes up
    assert L.orc_f64_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert L.orc_f64_to_bf16(1.0 + 2.0 ** -8 - 2.0 ** -40) == 0x3F80
    assert L.orc_f64_to_bf16(-(1.0 + 3 * 2.0 ** -8)) == 0xBF82
    assert L.orc_f64_to_bf16(0.0) == 0 and L.orc_f64_to_bf16(-0.0) == 0x8000
    assert L.orc_f64_to_bf16(1e300) == 0x7F80
