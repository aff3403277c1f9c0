"""Pins of the oracle's NVFP4 quantiser (block-scale / decode equation of the
miniTE Technical Report section 5.1; per-token and per-row outer scales of
its section 4.3 table and of the rainbus summary, method step 4)."""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(a):
    import synth
    return synth.to_bf16_bits(np.asarray(a, np.float32))


def _f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def load_worked_example():
    xs, exp = [], {}
    with open(os.path.join(GOLDEN, "nvfp4_worked_example.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "x":
                xs += [float(v) for v in vals]
            elif key == "g":
                exp["g"] = float(vals[0])
            else:
                exp[key] = [int(v, 16) for v in vals]
    return np.array(xs, np.float32), exp


def test_worked_example(orc):
    x, exp = load_worked_example()
    # the fixture's inputs are exact BF16 values
    assert np.array_equal(_f32(_bf16(x)), x)
    codes, sf, g = orc.quantize_row(x)
    assert g == exp["g"]
    assert list(sf) == exp["sf"]
    assert list(codes) == exp["codes"]
    # the same row, padded with a fourth zero block to K = 64, through the
    # batched BF16 path with swizzled scales
    x64 = np.concatenate([x, np.zeros(16, np.float32)])
    c2, s2, g2 = orc.quantize_rows(_bf16(x64)[None, :])
    assert list(c2[0]) == exp["codes"] + [0] * 8 and g2[0] == exp["g"]
    assert list(orc.unswizzle_sf(s2, 1, 64)[0]) == exp["sf"] + [0]


def test_zero_row(orc):
    codes, sf, g = orc.quantize_row(np.zeros(64, np.float32))
    assert g == 0.0 and not codes.any() and not sf.any()
    codes, sf, g = orc.quantize_row(np.array([-0.0] * 64, np.float32))
    assert g == 0.0 and not codes.any()


def _lossless_rows(rng, rows, K, g_exp):
    """Rows x = g s_b c with power-of-two g, one element 6*448*g per row and
    one element 6 s_b g per block, so that every quotient is exact."""
    g = 2.0 ** g_exp
    e4m3_vals = np.array([2.0 ** e * (1 + m / 8) for e in range(-6, 9) for m in range(8)
                          if 2.0 ** e * (1 + m / 8) <= 448])
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6])
    x = np.zeros((rows, K))
    for r in range(rows):
        for b in range(K // 16):
            s = 448.0 if b == 0 else rng.choice(e4m3_vals)
            blk = rng.choice(grid, 16)
            blk[rng.integers(16)] = 6.0 * rng.choice([1, -1])
            x[r, b * 16:(b + 1) * 16] = blk * s * g
    return x.astype(np.float32)


@pytest.mark.parametrize("g_exp", [-12, -3, 0, 4])
def test_lossless_rows_reconstruct_exactly(orc, g_exp):
    rng = np.random.default_rng(g_exp + 100)
    K = 128
    x = _lossless_rows(rng, 6, K, g_exp)
    xb = _bf16(x)
    assert np.array_equal(_f32(xb), x)
    codes, sf, g = orc.quantize_rows(xb)
    xh = orc.dequantize_rows(codes, sf, g, K)
    assert np.array_equal(xh, x.astype(np.float64))
    assert np.all(g == np.float32(2.0 ** g_exp))


def test_reconstruction_identity_and_error_bound(orc):
    """x^ = g s_b c, and every element is within half an E2M1 step of x
    (in units of its block scale), or saturated at 6."""
    rng = np.random.default_rng(5)
    K = 256
    x = rng.standard_normal((32, K)).astype(np.float32)
    x[:, 7] *= 50.0
    xb = _bf16(x)
    xv = _f32(xb).astype(np.float64)
    codes, sfs, g = orc.quantize_rows(xb)
    sf = orc.unswizzle_sf(sfs, 32, K)
    xh = orc.dequantize_rows(codes, sfs, g, K)
    e4m3 = np.array([orc.e4m3_value(c) for c in range(256)], np.float64)
    for r in range(32):
        S = np.repeat(np.float32(g[r]) * e4m3[sf[r]].astype(np.float32), 16).astype(np.float64)
        q = xv[r] / S
        aq = np.abs(q)
        gap = np.where(aq < 2, 0.5, np.where(aq < 4, 1.0, 2.0))
        err = np.abs(xh[r] - xv[r]) / S
        bound = np.maximum(gap / 2, aq - 6.0) * (1 + 1e-6) + 1e-12
        assert np.all(err <= bound)
    # amax of the row is represented within its block's rounding (scale 448)
    assert np.all(np.abs(np.abs(xh).max(1) - np.abs(xv).max(1)) <= np.abs(xv).max(1) / 12 + 1e-12)


def test_relative_error_matches_pages_order_of_magnitude(orc):
    """The pages report rel-L2 about 0.10 and SNR about 20 dB for E2M1 with
    E4M3 block scales (Technical Report section 2.3 format tables).  Gaussian
    rows give the same order of magnitude."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((64, 1024)).astype(np.float32)
    xb = _bf16(x)
    xv = _f32(xb).astype(np.float64)
    codes, sf, g = orc.quantize_rows(xb)
    xh = orc.dequantize_rows(codes, sf, g, 1024)
    rel = np.linalg.norm(xh - xv) / np.linalg.norm(xv)
    snr = 20 * np.log10(1 / rel)
    assert 0.07 < rel < 0.15, rel
    assert 16 < snr < 23


def test_given_amax_and_row_map(orc):
    rng = np.random.default_rng(3)
    src = _bf16(rng.standard_normal((5, 64)))
    rm = np.array([2, -1, 0, 4, 4, -1, 1], np.int32)
    am = orc.amax_rows(src)
    c1, s1, g1 = orc.quantize_rows(src, rm, am)
    c2, s2, g2 = orc.quantize_rows(src, rm, None)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2) and np.array_equal(g1, g2)
    for r, s in enumerate(rm):
        if s < 0:
            assert not c1[r].any() and g1[r] == 0
            assert not orc.unswizzle_sf(s1, 7, 64)[r].any()
        else:
            c, sf, g = orc.quantize_row(_f32(src[s]))
            assert np.array_equal(c1[r], c) and g1[r] == g
            assert np.array_equal(orc.unswizzle_sf(s1, 7, 64)[r], sf)
    # a larger given amax changes g and the scales (amax is an input)
    c3, s3, g3 = orc.quantize_rows(src, None, am * 2)
    assert np.all(g3 == np.float32(am * 2) / np.float32(2688))


def test_amax_exact(orc):
    rng = np.random.default_rng(4)
    x = _bf16(rng.standard_normal((17, 96)) * 3)
    assert np.array_equal(orc.amax_rows(x), np.abs(_f32(x)).max(1))


def test_sf_layout_is_a_bijection_of_128x4_tiles(orc):
    """Every logical (row, col) maps to a distinct byte; a 512-byte tile holds
    exactly 128 rows x 4 columns; byte (r%32)*16 + ((r/32)%4)*4 + c%4."""
    rows, K = 256, 192
    offs = np.array([[orc.sf_offset(r, c, K) for c in range(K // 16)] for r in range(rows)])
    assert len(np.unique(offs)) == offs.size == orc.sf_bytes(rows, K)
    assert offs[0, 0] == 0 and offs[1, 0] == 16 and offs[32, 0] == 4 and offs[0, 1] == 1
    assert offs[0, 4] == 512 and offs[128, 0] == 512 * (K // 64)
    tiles = offs // 512
    for t in np.unique(tiles):
        rr, cc = np.nonzero(tiles == t)
        assert len(np.unique(rr)) == 128 and len(np.unique(cc)) == 4


def test_sf_layout_matches_tile_reshape(orc):
    """The block-scale layout built another way: a tile holds the scales of
    128 rows x 4 columns (4 blocks of 16 elements along K, one scale each)
    as a 32 x 16-byte array whose row i carries, for each of
    the row groups j = 0..3, the 4 column scales of row 32 j + i (the
    tensor core's block-scale tile: each of the 32 lanes of a 32-row quadrant
    reads one 16-byte row).  Tiles follow row block by row block, column
    group fastest.  Built here by reshaping the logical [rows][K/16] array,
    not from the oracle's offset formula, and compared through the oracle's
    unswizzle."""
    rng = np.random.default_rng(21)
    rows, K = 256, 192
    logical = rng.integers(0, 256, size=(rows, K // 16), dtype=np.uint8)
    tiles = []
    for b in range(rows // 128):
        for g in range(K // 64):
            t = logical[128 * b:128 * (b + 1), 4 * g:4 * (g + 1)]  # [128 rows][4 columns]
            tiles.append(t.reshape(4, 32, 4).transpose(1, 0, 2).reshape(512))  # [lane i][group j][column c]
    buf = np.concatenate(tiles)
    assert buf.size == orc.sf_bytes(rows, K)
    assert np.array_equal(orc.unswizzle_sf(buf, rows, K), logical)


def test_context_swap_invariance(orc):
    """Per-token scales: a row's codes, scales and outer scale do not depend on
    the other rows of the batch (the context-swap property of the AI summary's
    methodology section)."""
    rng = np.random.default_rng(9)
    x = _bf16(rng.standard_normal((8, 128)))
    c0, s0, g0 = orc.quantize_rows(x)
    y = x.copy()
    y[[0, 1, 2, 4, 5, 6, 7]] = _bf16(rng.standard_normal((7, 128)) * 100)
    y = y[[3, 0, 1, 2, 4, 5, 6, 7]]  # target row 3 moves to position 0
    c1, s1, g1 = orc.quantize_rows(y)
    assert np.array_equal(c1[0], c0[3]) and g1[0] == g0[3]
    assert np.array_equal(orc.unswizzle_sf(s1, 8, 128)[0], orc.unswizzle_sf(s0, 8, 128)[3])
