"""Pins of the oracle's contrast recipes (not the hot path's recipe).

* The blockwise random Hadamard transform is the Sylvester Hadamard matrix
  of scipy, scaled by 1/4 and signed per column, and is its own inverse up
  to the sign vector (orthogonality).
* Per-tensor quantisation is per-row quantisation with the tensor's amax.
* The context-swap contrast the miniTE summary reports ("Methodology in
  Plain English"): with per-token scales a target row's codes are bitwise
  unchanged when the other tokens of its batch are replaced, while an
  RHT-enabled per-tensor reference changes them.
* Per-expert weight scales ("miniTE CUTLASS" column of the Technical
  Report's section 4.3 table): one g per expert tensor, reducing to the
  per-row recipe when every row of the expert has the same amax.
"""
import numpy as np
import pytest

from helpers import bf16, f32


def _signs(seed=7):
    rng = np.random.default_rng(seed)
    return np.where(rng.random(16) < 0.5, -1, 1).astype(np.int8)


def test_rht_is_scaled_signed_sylvester_hadamard(orc):
    sl = pytest.importorskip("scipy.linalg")
    H = sl.hadamard(16).astype(np.float64)
    s = _signs()
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 64)).astype(np.float32)
    y = orc.rht16_rows(x, s)
    ref = np.empty_like(y)
    for r in range(5):
        for b in range(4):
            blk = x[r, 16 * b:16 * b + 16].astype(np.float64) * s
            ref[r, 16 * b:16 * b + 16] = (0.25 * (H @ blk)).astype(np.float32)
    assert np.allclose(y, ref, rtol=2e-7, atol=1e-30)
    # basis vectors map exactly onto signed, scaled Hadamard columns
    e = np.eye(16, dtype=np.float32)
    ye = orc.rht16_rows(e, s)
    assert np.array_equal(ye, (0.25 * H * s[None, :]).T.astype(np.float32))


def test_rht_is_orthogonal(orc):
    s = _signs(3)
    rng = np.random.default_rng(2)
    x = rng.standard_normal((8, 128)).astype(np.float32)
    y = orc.rht16_rows(x, s).astype(np.float64)
    sl = pytest.importorskip("scipy.linalg")
    H = sl.hadamard(16).astype(np.float64)
    back = np.empty_like(y)
    for b in range(8):
        back[:, 16 * b:16 * b + 16] = 0.25 * (y[:, 16 * b:16 * b + 16] @ H) * s[None, :]
    assert np.allclose(back, x, rtol=0, atol=1e-6 * np.abs(x).max())
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x.astype(np.float64), axis=1), rtol=1e-6)


def test_per_tensor_is_row_quantisation_with_the_tensor_amax(orc):
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((6, 64)) * np.array([0.1, 1, 3, 0.5, 10, 2])[:, None]).astype(np.float32)
    codes, sf, g = orc.quantize_tensor(x)
    a = float(np.abs(x).max())
    assert np.all(g == g[0]) and g[0] == np.float32(a) / np.float32(2688.0)
    logical = orc.unswizzle_sf(sf, 6, 64)
    for r in range(6):
        c, s_, gr = orc.quantize_row(x[r], amax=a)
        assert np.array_equal(codes[r], c) and np.array_equal(logical[r], s_) and gr == g[r]


def test_context_swap_contrast(orc):
    """Six swaps of the other tokens of a batch against a reference batch: the
    per-token codes of the target row never change; the RHT-enabled
    per-tensor reference's change whenever another token raises the tensor's
    amax (the summary reports five of six swaps)."""
    rng = np.random.default_rng(11)
    d = 256
    target = bf16(rng.standard_normal(d).astype(np.float32))
    s = _signs(5)

    def codes_of_target(other_scale, seed):
        others = bf16((np.random.default_rng(seed).standard_normal((7, d)) * other_scale).astype(np.float32))
        batch = np.concatenate([target[None, :], others])
        c_tok, sf_tok, g_tok = orc.quantize_rows(batch)
        c_rht, sf_rht, g_rht = orc.quantize_per_tensor_rht(batch, s)
        tok = (c_tok[0].tobytes(), orc.unswizzle_sf(sf_tok, 8, d)[0].tobytes(), float(g_tok[0]))
        rht = (c_rht[0].tobytes(), orc.unswizzle_sf(sf_rht, 8, d)[0].tobytes(), float(g_rht[0]))
        return tok, rht

    ref_tok, ref_rht = codes_of_target(0.25, 99)
    changed_tok = changed_rht = 0
    for i, sc in enumerate([0.5, 2.0, 4.0, 8.0, 16.0, 32.0]):
        tok, rht = codes_of_target(sc, 100 + i)
        changed_tok += tok != ref_tok
        changed_rht += rht != ref_rht
    assert changed_tok == 0
    assert changed_rht >= 4


def test_per_expert_weight_scale(orc):
    rng = np.random.default_rng(21)
    E, N, K = 3, 8, 64
    # rows spanning four decades: under one shared scale the small rows'
    # block scales fall into the E4M3 subnormal range
    W = bf16((rng.standard_normal((E, N, K)) * 10.0 ** rng.uniform(-4.0, 0.5, (E, N, 1)) * 0.02).astype(np.float32))
    codes, sf, g = orc.quantize_weights_per_expert(W)
    logical = orc.unswizzle_sf(sf, E * N, K)
    for e in range(E):
        a = float(np.abs(f32(W[e])).max())
        assert np.all(g[e] == np.float32(a) / np.float32(2688.0))
        for n in range(N):
            c, s_, gr = orc.quantize_row(f32(W[e, n]), amax=a)
            assert np.array_equal(codes[e, n], c) and np.array_equal(logical[e * N + n], s_)
    # rows sharing one amax: identical to the per-row recipe
    Weq = np.array(W)
    Weq[:, :, 0] = bf16(np.float32(0.25))  # every row's max |w| is 0.25
    Weq[:, :, 1:] = bf16((f32(W[:, :, 1:]) / (np.abs(f32(W)).max() * 8)).astype(np.float32))
    c1, s1, g1 = orc.quantize_weights_per_expert(Weq)
    c2, s2, g2 = orc.quantize_weights(Weq)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2) and np.array_equal(g1, g2)
    # varying row scales: the shared scale reconstructs worse
    rec_e = orc.dequantize_rows(codes.reshape(E * N, K // 2), sf, g.reshape(-1), K)
    cr, sr, gr_ = orc.quantize_weights(W)
    rec_r = orc.dequantize_rows(cr.reshape(E * N, K // 2), sr, gr_.reshape(-1), K)
    ref = f32(W).reshape(E * N, K).astype(np.float64)
    assert np.linalg.norm(rec_e - ref) > np.linalg.norm(rec_r - ref)
