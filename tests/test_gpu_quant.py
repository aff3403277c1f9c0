"""Bit-exact parity of the GPU quantisers with the oracle: codes, block
scales (compared after un-swizzling with the oracle's layout) and outer
scales, for weights, activation rows, row maps, given amax and pad rows."""
import numpy as np
import pytest

import nvfp4_w4a4_moe_top_gb300 as M
import synth
from helpers import bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from nvfp4_w4a4_moe_top_gb300 import build
    build.build()


def _cmp(orc, got, exp, rows, K):
    gc, gs, gg = got
    ec, es, eg = exp
    assert np.array_equal(gc[:rows], ec[:rows])
    assert np.array_equal(gg[:rows].view(np.uint32), eg[:rows].view(np.uint32))
    assert np.array_equal(orc.unswizzle_sf(gs, rows, K), orc.unswizzle_sf(es, rows, K))


# scale 1e36: row maxima near 1e38, outer scales above 2^111, and the row
# near 1e-38 below 2^-87: rows the main pass leaves to the fix-up pass
@pytest.mark.parametrize("rows,K,scale", [(1, 64, 1.0), (37, 128, 1.0), (300, 768, 3.0), (129, 2048, 0.02),
                                          (64, 4096, 1.0), (200, 1024, 1e-3), (50, 256, 1e30), (40, 2048, 1e36)])
def test_quantize_rows_bitexact(orc, rows, K, scale):
    from gpu_util import dev, host
    import torch
    rng = np.random.default_rng(rows * K)
    x = rng.standard_normal((rows, K)) * scale
    x[:, rng.integers(K, size=3)] *= 40
    x[rows // 2] = 0.0                        # all-zero row
    if rows > 3:
        x[1, :] = rng.standard_normal(K) * 1e-38   # subnormal-range row
        x[2, :16] = 0.0                        # zero block
    xb = bf16(x)
    q = M.empty_quantized(rows, K)
    M.nvfp4_quantize_rows(dev(xb), K, None, None, rows, q["codes"], q["sf"], q["g"])
    torch.cuda.synchronize()
    got = (host(q["codes"]), host(q["sf"]), host(q["g"]))
    _cmp(orc, got, orc.quantize_rows(xb), rows, K)


@pytest.mark.parametrize("g_exp", [-14, -3, 2])
def test_quantize_rows_exact_ties(orc, g_exp):
    """Rows built from exact block scales and E2M1 grid values and midpoints:
    every quotient is exact, half of them exact rounding ties, which the
    quantiser must resolve like the specification (nearest even)."""
    from gpu_util import dev, host
    from helpers import lossless_rows
    import torch
    rng = np.random.default_rng(50 + g_exp)
    rows, K = 96, 256
    x = lossless_rows(rng, rows, K, g_exp)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    # replace a third of the non-maximal elements by midpoints (ties)
    blk = np.abs(x).reshape(rows, K // 16, 16).max(2, keepdims=True) / 6.0
    sel = rng.random(x.shape) < 0.33
    m = rng.choice(mids, x.shape) * rng.choice([-1, 1], x.shape)
    tied = (m.reshape(rows, K // 16, 16) * blk).reshape(rows, K)
    x = np.where(sel & (np.abs(x) < np.repeat(blk.reshape(rows, -1), 16, 1) * 6), tied, x).astype(np.float32)
    xb = bf16(x)
    q = M.empty_quantized(rows, K)
    M.nvfp4_quantize_rows(dev(xb), K, None, None, rows, q["codes"], q["sf"], q["g"])
    torch.cuda.synchronize()
    _cmp(orc, (host(q["codes"]), host(q["sf"]), host(q["g"])), orc.quantize_rows(xb), rows, K)


def test_quantize_rows_map_amax_and_pad(orc):
    from gpu_util import dev, host
    import torch
    rng = np.random.default_rng(7)
    K, src_rows = 512, 40
    xb = bf16(rng.standard_normal((src_rows, K)))
    rm = rng.integers(-1, src_rows, 300).astype(np.int32)
    am = orc.amax_rows(xb) * np.float32(1.5)
    for amax in [None, am]:
        q = M.empty_quantized(300, K)
        M.nvfp4_quantize_rows(dev(xb), K, dev(rm), None if amax is None else dev(amax), 300,
                              q["codes"], q["sf"], q["g"])
        torch.cuda.synchronize()
        got = (host(q["codes"]), host(q["sf"]), host(q["g"]))
        _cmp(orc, got, orc.quantize_rows(xb, rm, amax, 300), 300, K)


def test_quantize_weights_bitexact(orc):
    from gpu_util import dev, host
    import torch
    lay = synth.layer("small")
    W1 = np.stack([lay.w1_expert(e) for e in range(3)])
    W2 = np.stack([lay.w2_expert(e) for e in range(3)])
    for W in (W1, W2):
        q = M.quantize_weights(dev(W))
        torch.cuda.synchronize()
        E, N, K = W.shape
        ec, es, eg = orc.quantize_weights(W)
        assert np.array_equal(host(q["codes"]), ec)
        assert np.array_equal(host(q["g"]).view(np.uint32), eg.view(np.uint32))
        assert np.array_equal(orc.unswizzle_sf(host(q["sf"]), E * N, K), orc.unswizzle_sf(es, E * N, K))


def test_nonfinite_sets_status(orc):
    from gpu_util import dev, host
    import torch
    x = np.zeros((8, 64), np.float32)
    x[3, 5] = np.inf
    x[6, 1] = np.nan
    q = M.empty_quantized(8, 64)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.nvfp4_quantize_rows(dev(bf16(x)), 64, None, None, 8, q["codes"], q["sf"], q["g"], st)
    torch.cuda.synchronize()
    assert int(st.item()) & M.STATUS_NONFINITE_X
    W = np.zeros((1, 128, 64), np.float32)
    W[0, 7, 7] = np.nan
    st.zero_()
    q = M.empty_quantized(128, 64)
    M.moe_nvfp4_quantize_weights(dev(bf16(W)), q["codes"], q["sf"], q["g"], st)
    torch.cuda.synchronize()
    assert int(st.item()) & M.STATUS_NONFINITE_WEIGHT


def test_guard_bytes_untouched(orc):
    from gpu_util import dev, host
    import torch
    rows, K = 130, 192
    xb = bf16(np.random.default_rng(1).standard_normal((rows, K)))
    G = 4096
    codes = torch.full((rows * K // 2 + G,), 0xA5, dtype=torch.uint8, device="cuda")
    sfb = M.sf_bytes(rows, K)
    sf = torch.full((sfb + G,), 0xA5, dtype=torch.uint8, device="cuda")
    g = torch.full((rows + G,), 7.0, dtype=torch.float32, device="cuda")
    M.nvfp4_quantize_rows(dev(xb), K, None, None, rows, codes, sf, g)
    torch.cuda.synchronize()
    assert np.all(host(codes)[rows * K // 2:] == 0xA5)
    assert np.all(host(sf)[sfb:] == 0xA5)
    assert np.all(host(g)[rows:] == 7.0)
