"""Pins of the oracle's router, permutation, grouped GEMM and epilogues.

Router and permutation are checked against library sorts and softmax; the
grouped GEMM against an FP64 matmul of the dequantised operands (an exact
dot product within the FP32 summation bound); SwiGLU, the router-weighted
cast and the reduce against closed forms and torch's BF16 cast.
"""
import numpy as np
import pytest
import scipy.special
import torch


def _bf16(a):
    import synth
    return synth.to_bf16_bits(np.asarray(a, np.float32))


def _f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _torch_bf16(x32):
    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


# ---- router -----------------------------------------------------------------
@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (50, 32, 4), (20, 128, 8), (7, 5, 5), (9, 16, 1)])
def test_route_matches_library_sort_and_softmax(orc, T, E, k):
    rng = np.random.default_rng(T * E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[0, :] = 0.5                      # an all-tie row: lowest ids win
    lg[1, 3:] = lg[1, 2]                # partial ties
    ids, w = orc.route(lg, k)
    for t in range(T):
        order = np.lexsort((np.arange(E), -lg[t].astype(np.float64)))
        sel = np.sort(order[:k])
        assert np.array_equal(ids[t], sel)
        ref = scipy.special.softmax(lg[t, sel].astype(np.float64))
        assert np.allclose(w[t], ref, rtol=2e-7, atol=0)
        # softmax over all experts, then top-k, then renormalise: same weights
        full = scipy.special.softmax(lg[t].astype(np.float64))
        ren = full[sel] / full[sel].sum()
        assert np.allclose(w[t], ren, rtol=1e-6, atol=0)
    assert np.array_equal(ids[0], np.arange(k))


def test_route_rejects_nonfinite(orc):
    lg = np.zeros((2, 8), np.float32)
    lg[1, 3] = np.nan
    with pytest.raises(ValueError):
        orc.route(lg, 2)


# ---- permutation ------------------------------------------------------------
def _perm_invariants(perm, ids, E):
    T, k = ids.shape
    c, off, r2t, tsr = perm["counts"], perm["offsets"], perm["row_to_token"], perm["token_slot_row"]
    assert c.sum() == T * k
    assert np.array_equal(c, np.bincount(ids.ravel(), minlength=E))
    assert off[0] == 0 and np.all(off % 128 == 0) and off[E] == perm["m_pad"]
    assert np.array_equal(np.diff(off), (c + 127) // 128 * 128)
    assert perm["m_pad"] <= perm["m_cap"] and perm["m_cap"] % 128 == 0
    used = np.zeros(perm["m_cap"], bool)
    for t in range(T):
        for j in range(k):
            r = tsr[t, j]
            e = ids[t, j]
            assert off[e] <= r < off[e] + c[e]
            assert r2t[r] == t and not used[r]
            used[r] = True
    assert np.all((r2t >= 0) == used)
    for e in range(E):
        rows = r2t[off[e]:off[e] + c[e]]
        assert np.all(np.diff(rows) > 0)          # ascending tokens per expert
        assert np.all(r2t[off[e] + c[e]:off[e + 1]] == -1)


@pytest.mark.parametrize("T,E,k,skew", [(256, 8, 2, 0), (300, 32, 4, 3.0), (97, 128, 8, 2.0), (1, 4, 4, 0)])
def test_permute_invariants_and_library_sort(orc, T, E, k, skew):
    rng = np.random.default_rng(T + E)
    lg = rng.standard_normal((T, E)) + skew * rng.standard_normal(E)[None, :]
    ids, _ = orc.route(lg.astype(np.float32), k)
    perm = orc.permute(ids, E)
    _perm_invariants(perm, ids, E)
    # brute force: a stable sort of (expert, token) pairs by expert
    flat_e = ids.ravel()
    order = np.argsort(flat_e, kind="stable")
    tok = np.repeat(np.arange(T), k)
    for e in range(E):
        got = perm["row_to_token"][perm["offsets"][e]:perm["offsets"][e] + perm["counts"][e]]
        assert np.array_equal(got, tok[order[flat_e[order] == e]])


def test_permute_empty_experts(orc):
    ids = np.array([[0, 3], [0, 3], [3, 5]], np.int32)
    perm = orc.permute(ids, 8)
    _perm_invariants(perm, ids, 8)
    assert list(perm["offsets"]) == [0, 128, 128, 128, 256, 256, 384, 384, 384]
    assert perm["m_pad"] == 384


# ---- grouped GEMM -----------------------------------------------------------
def _quantize(orc, rng, rows, K, scale=1.0):
    x = _bf16(rng.standard_normal((rows, K)) * scale)
    return x, orc.quantize_rows(x)


@pytest.mark.parametrize("E,K,N", [(1, 64, 64), (2, 128, 64), (3, 64, 128)])
def test_grouped_gemm_against_fp64_matmul(orc, E, K, N):
    rng = np.random.default_rng(E * K + N)
    counts = [5, 0, 9][:E]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(off[-1])
    _, (ac, asf, ag) = _quantize(orc, rng, M, K)
    W = _bf16(rng.standard_normal((E * N, K)) * 0.02)
    wc, wsf, wg = orc.quantize_rows(W)
    y = orc.grouped_gemm(ac, asf, ag, off, wc.reshape(E, N, K // 2), wsf, wg.reshape(E, N), K, N)
    A = orc.dequantize_rows(ac, asf, np.ones_like(ag), K)      # c_a s_a
    B = orc.dequantize_rows(wc, wsf, np.ones_like(wg), K)      # c_w s_w
    for e in range(E):
        for r in range(off[e], off[e + 1]):
            Be = B[e * N:(e + 1) * N]
            exact = Be @ A[r]
            bound = K * 2.0 ** -24 * (np.abs(Be) @ np.abs(A[r]))
            acc = y[r] / (np.float32(ag[r]) * wg[e * N:(e + 1) * N]).astype(np.float64)
            ok = np.abs(acc - exact) <= bound * 1.01 + 1e-30
            assert np.all(ok | (ag[r] * wg[e * N:(e + 1) * N] == 0))
            # the epilogue scales by (g_a g_w) formed first, in FP32
            scale = (np.float32(ag[r]) * wg[e * N:(e + 1) * N]).astype(np.float32)
            assert np.all(np.isfinite(y[r])) and np.all(np.abs(y[r]) <= np.abs(exact * scale) + bound * scale * 1.01 + 1e-30)


def test_single_expert_reduces_to_dense_gemm(orc):
    """E = 1: the grouped GEMM is one dense GEMM of the dequantised operands."""
    rng = np.random.default_rng(2)
    K, N, M = 256, 96, 40
    _, (ac, asf, ag) = _quantize(orc, rng, M, K)
    W = _bf16(rng.standard_normal((N, K)))
    wc, wsf, wg = orc.quantize_rows(W)
    y = orc.grouped_gemm(ac, asf, ag, np.array([0, M], np.int32), wc[None], wsf, wg[None], K, N)
    ref = orc.dequantize_rows(ac, asf, ag, K) @ orc.dequantize_rows(wc, wsf, wg, K).T
    assert np.allclose(y, ref, rtol=1e-5, atol=1e-5 * np.abs(ref).max())


def test_lossless_operands_give_the_bf16_gemm(orc):
    """Rows exactly representable in NVFP4 quantise losslessly, so the GEMM
    equals the GEMM of the original BF16 values (within FP32 summation)."""
    from helpers import lossless_rows
    rng = np.random.default_rng(21)
    K, N, M = 128, 32, 16
    x = lossless_rows(rng, M, K, -11)
    w = lossless_rows(rng, N, K, -14)
    xb, wb = _bf16(x), _bf16(w)
    ac, asf, ag = orc.quantize_rows(xb)
    wc, wsf, wg = orc.quantize_rows(wb)
    assert np.array_equal(orc.dequantize_rows(ac, asf, ag, K), _f32(xb).astype(np.float64))
    y = orc.grouped_gemm(ac, asf, ag, np.array([0, M], np.int32), wc[None], wsf, wg[None], K, N)
    X, Wm = _f32(xb).astype(np.float64), _f32(wb).astype(np.float64)
    ref = X @ Wm.T
    bound = K * 2.0 ** -23 * (np.abs(X) @ np.abs(Wm).T)
    assert np.all(np.abs(y - ref) <= bound + 1e-30)


# ---- epilogues --------------------------------------------------------------
def test_swiglu_is_correctly_rounded_silu_times_up(orc):
    rng = np.random.default_rng(8)
    F = 64
    y = (rng.standard_normal((16, 2 * F)) * 4).astype(np.float32)
    y[0, :F] = 0.0
    y[1, :F] = 80.0
    u, h = orc.swiglu(y, F)
    assert np.array_equal(u, _torch_bf16(y))
    zg = _f32(u[:, :F]).astype(np.float64)
    zu = _f32(u[:, F:]).astype(np.float64)
    ref = zg * scipy.special.expit(zg) * zu
    hv = _f32(h).astype(np.float64)
    # correctly rounded: within half a BF16 ulp of the exact value
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-38))) - 7)
    assert np.all(np.abs(hv - ref) <= 0.5 * ulp * (1 + 1e-9) + 1e-300)
    assert np.all(hv[0] == 0)                          # silu(0) = 0
    assert np.array_equal(h[1], _torch_bf16(np.float32(80.0) * _f32(u[1, F:])))


def test_combine_and_reduce(orc):
    rng = np.random.default_rng(12)
    T, k, d = 6, 3, 32
    ids = np.array([[0, 1, 2]] * T, np.int32)
    perm = orc.permute(ids, 3)
    y2 = (rng.standard_normal((perm["m_cap"], d))).astype(np.float32)
    w = rng.random((T, k)).astype(np.float32)
    slots = orc.combine(y2, perm, w, T, k, d)
    for t in range(T):
        for j in range(k):
            r = perm["token_slot_row"][t, j]
            assert np.array_equal(slots[t, j], _torch_bf16(w[t, j] * y2[r]))
    out = orc.reduce(slots)
    s = _f32(slots[:, 0]).copy()
    for j in range(1, k):
        s = (s + _f32(slots[:, j])).astype(np.float32)
    assert np.array_equal(out, _torch_bf16(s))
    # k = 1: the reduce is the identity on BF16 values
    assert np.array_equal(orc.reduce(slots[:, :1]), slots[:, 0])


def test_reduce_order_is_ascending_slot(orc):
    """FP32 addition is not associative, so the slot order is observable:
    256 + 1 = 257 is a BF16 midpoint; adding 2^-16 twice afterwards is
    absorbed (FP32 ties to even), while 2^-16 + 2^-16 + 1 + 256 lands just
    above the midpoint and rounds up."""
    a, b, c = 256.0, 1.0, 2.0 ** -16
    s1 = _bf16(np.array([[[a], [b], [c], [c]]], np.float32))
    s2 = _bf16(np.array([[[c], [c], [b], [a]]], np.float32))
    assert _f32(orc.reduce(s1))[0, 0] == 256.0
    assert _f32(orc.reduce(s2))[0, 0] == 258.0
