"""End-to-end parity of moe_expert_forward (the call bench.py times).

Against the fully independent oracle: routing, permutation, offsets and the
activation codes / scales / outer scales are bit-exact; h codes and the BF16
output agree within the tolerance that the tensor-core accumulation order
allows (see the stage-wise checks in test_gpu_gemm.py).  The fused forward
equals the composition of the modular entry points bit for bit, is
deterministic, flags non-finite inputs, and leaves memory outside its
outputs untouched.  At the Qwen-shaped sizes, sampled tokens are checked one
by one against the oracle.
"""
import numpy as np
import pytest

import nvfp4_w4a4_moe_top_gb300 as M
import synth
from helpers import bf16

pytestmark = pytest.mark.gpu

# Independent end-to-end tolerance on the BF16 output.  The FP32 sums of the
# GEMMs run in the tensor cores' order, not the oracle's sequential order
# (about 1e-7 relative); with h rounded exactly on both sides, what reaches
# the output is a rare flip of a BF16 rounding: of u (which can move an h
# code), of one of the token's k slot values z = BF16(w y2), or of out itself.
# Per element, then, out may differ from the oracle's by at most one BF16 ulp
# of out plus one BF16 ulp of each of the k slot values (the oracle's) that
# were summed into it: where the slots cancel, that is several ulps of out.
# Measured on GB300 over the configurations below: rel-L2 at most 1.1e-5,
# at most 0.5 of that per-element bound, no h-code row different.  The
# checks: rel-L2 <= 2e-5, every element within the bound, h-code rows
# differing <= 1e-3.
E2E_REL_L2 = 2e-5
H_ROWS_DIFFERING = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from nvfp4_w4a4_moe_top_gb300 import build
    build.build()


def gpu_forward(lay, x, lg, W1=None, W2=None, w1q=None, w2q=None, status=True):
    import torch
    from gpu_util import dev, host
    T, E, k, d, dff = x.shape[0], lay.E, lay.k, lay.d, lay.d_ff
    if w1q is None:
        w1q = M.quantize_weights(dev(W1))
        w2q = M.quantize_weights(dev(W2))
    out = torch.full((T, d), 0x5A5A, dtype=torch.int16, device="cuda")
    ws = M.forward_workspace(T, E, k, d, dff)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_expert_forward(dev(x), dev(lg), T, E, k, d, dff, w1q["codes"], w1q["sf"], w1q["g"], w2q["codes"],
                         w2q["sf"], w2q["g"], out, ws, st)
    torch.cuda.synchronize()
    v = M.forward_views(ws, T, E, k, d, dff)
    r = {n: (host(t) if hasattr(t, "cpu") else t) for n, t in v.items()}
    r["out"] = host(out, np.uint16)
    r["status"] = int(st.item())
    r["ws"] = ws
    return r, w1q, w2q


def bf16_ulp(v):
    """Spacing of BF16 values at |v| (v in FP32)."""
    return np.ldexp(1.0, np.frexp(np.maximum(np.abs(v), 2.0 ** -126))[1] - 8)


def e2e_errors(got_bf16, exp_bf16, slots_bf16):
    """rel-L2, max-abs, and the largest ratio of |got - expected| to the
    per-element bound ulp(expected) + sum_j ulp(z_j), z_j the oracle's k slot
    values [T][k][d] behind each output element."""
    from gpu_util import f32_of_bf16, rel_l2
    g, e = f32_of_bf16(got_bf16), f32_of_bf16(exp_bf16)
    bound = bf16_ulp(e) + bf16_ulp(f32_of_bf16(slots_bf16)).sum(axis=1)
    return rel_l2(g, e), float(np.abs(g - e).max()), float((np.abs(g - e) / bound).max())


def layer_of(name):
    if name == "ragged":
        return synth.custom(T=999, d=384, E=12, k=3, d_ff=256, seed=11, logits="bias", bias_std=2.0,
                            n_forced_empty=3)
    if name == "k1":
        return synth.custom(T=130, d=256, E=4, k=1, d_ff=128, seed=2)
    if name == "single_expert":
        return synth.custom(T=200, d=128, E=1, k=1, d_ff=128, seed=3)
    if name == "all_experts":
        return synth.custom(T=64, d=256, E=6, k=6, d_ff=256, seed=8)
    if name == "max_experts":  # E and k at their limits: ~2 rows per expert, mostly pad rows
        return synth.custom(T=64, d=128, E=1024, k=32, d_ff=128, seed=13)
    if name == "max_width":  # d and d_ff at their limits: A streams through the stages in both GEMMs
        return synth.custom(T=160, d=4096, E=2, k=1, d_ff=4096, seed=14)
    if name == "ragged_pairs":  # FC2 on CTA pairs (three rings) with empty experts and odd tile counts
        return synth.custom(T=1500, d=512, E=12, k=3, d_ff=256, seed=13, logits="bias", bias_std=2.0,
                            n_forced_empty=3)
    return synth.layer(name)


@pytest.mark.parametrize("name", ["tiny", "small", "ragged", "k1", "single_expert", "all_experts", "max_experts",
                                  "max_width"])
def test_forward_against_oracle(orc, name):
    lay = layer_of(name)
    x, lg, W1, W2 = lay.x(), lay.logits(), lay.w1(), lay.w2()
    r, _, _ = gpu_forward(lay, x, lg, W1, W2)
    assert r["status"] == 0
    ref = orc.moe_forward(x, lg, orc.quantize_weights(W1), orc.quantize_weights(W2), lay.k, lay.d_ff)
    perm = ref["perm"]
    mp = perm["m_pad"]
    assert np.array_equal(r["topk_ids"], ref["ids"])
    assert np.allclose(r["topk_w"], ref["w"], rtol=1e-6, atol=0)
    for key in ["counts", "offsets", "row_to_token", "token_slot_row"]:
        assert np.array_equal(r[key], perm[key]), key
    assert np.array_equal(r["amax_tok"].view(np.uint32), ref["amax_tok"].view(np.uint32))
    assert np.array_equal(r["x_codes"][:mp], ref["x_codes"][:mp])
    assert np.array_equal(r["x_g"][:mp].view(np.uint32), ref["x_g"][:mp].view(np.uint32))
    assert np.array_equal(orc.unswizzle_sf(r["x_sf"], mp, lay.d), orc.unswizzle_sf(ref["x_sf"], mp, lay.d))
    # h codes: identical except rows touched by a rare accumulation-order flip
    row_diff = np.any(r["h_codes"][:mp] != ref["h_codes"][:mp], axis=1)
    rel, mx, ratio = e2e_errors(r["out"], ref["out"], ref["slots"])
    print("%s: e2e rel-L2 %.3e max-abs %.3e (%.2f of the flip bound), h-code rows differing %.5f"
          % (name, rel, mx, ratio, row_diff.mean()))
    assert row_diff.mean() <= H_ROWS_DIFFERING, row_diff.mean()
    assert rel <= E2E_REL_L2 and ratio <= 1.0


def test_forward_extreme_token_scales(orc):
    """Tokens whose maxima are 4e-36 and 2e37 (outer scales outside
    [2^-87, 2^111]): the fused permute/quantise encodes them with the E2M1
    division's power-of-two row factor, bit-exact with the oracle's
    quantiser on the permuted rows.  The weights are scaled by 1e-36 (their
    outer scales also leave the range) so that every GEMM value stays
    finite; only the quantised x rows are compared."""
    from helpers import f32
    lay = layer_of("tiny")
    xf = f32(lay.x())
    peak = np.abs(xf).max(axis=1, keepdims=True)
    xf[0::7] *= 4e-36 / peak[0::7]
    xf[3::7] *= 2e37 / peak[3::7]
    x = bf16(xf)
    assert np.isfinite(f32(x)).all()
    W1, W2 = bf16(f32(lay.w1()) * 1e-36), bf16(f32(lay.w2()) * 1e-36)
    r, _, _ = gpu_forward(lay, x, lay.logits(), W1, W2)
    mp = int(r["offsets"][-1])
    codes, sf, g = orc.quantize_rows(x, row_map=r["row_to_token"][:mp], dst_rows=mp)
    assert np.array_equal(r["x_codes"][:mp], codes)
    assert np.array_equal(r["x_g"][:mp].view(np.uint32), g.view(np.uint32))
    assert np.array_equal(orc.unswizzle_sf(r["x_sf"], mp, lay.d), orc.unswizzle_sf(sf, mp, lay.d))
    gx = r["x_g"][:mp][r["row_to_token"][:mp] >= 0]
    assert (gx < 2.0 ** -87).any() and (gx > 2.0 ** 111).any()  # both sides of the range are exercised


@pytest.mark.parametrize("name", ["small", "ragged", "tiny", "ragged_pairs"])
def test_forward_cta_pairs_equal_single(orc, name, monkeypatch):
    """The forward with FC1 and FC2 on CTA pairs (the default where their
    shapes allow it) and with either GEMM on single CTAs: identical h codes
    and output, bit for bit."""
    lay = layer_of(name)
    x, lg, W1, W2 = lay.x(), lay.logits(), lay.w1(), lay.w2()
    r2, w1q, w2q = gpu_forward(lay, x, lg, W1, W2)
    runs = []
    for var in ("MOE_FC1_CTA_PAIRS", "MOE_FC2_CTA_PAIRS"):
        monkeypatch.setenv(var, "0")
        runs.append(gpu_forward(lay, x, lg, w1q=w1q, w2q=w2q)[0])
        monkeypatch.delenv(var)
    assert r2["status"] == 0 and all(r["status"] == 0 for r in runs)
    mp = int(r2["offsets"][-1])
    for r1 in runs:
        assert np.array_equal(r2["h_codes"][:mp], r1["h_codes"][:mp])
        assert np.array_equal(r2["h_g"][:mp].view(np.uint32), r1["h_g"][:mp].view(np.uint32))
        assert np.array_equal(r2["slots"][:mp], r1["slots"][:mp])
        assert np.array_equal(r2["out"], r1["out"])


def test_forward_equals_modular_composition(orc):
    """moe_expert_forward = moe_permute_amax + nvfp4_quantize_rows +
    FC1 + FC2/unpermute, bit for bit."""
    import torch
    from gpu_util import dev, host
    lay = synth.layer("small")
    x, lg, W1, W2 = lay.x(), lay.logits(), lay.w1(), lay.w2()
    T, E, k, d, dff = lay.T, lay.E, lay.k, lay.d, lay.d_ff
    r, w1q, w2q = gpu_forward(lay, x, lg, W1, W2)
    mc = M.m_cap(T, E, k)
    i32, f32 = torch.int32, torch.float32
    ids = torch.zeros((T, k), dtype=i32, device="cuda")
    w = torch.zeros((T, k), dtype=f32, device="cuda")
    counts = torch.zeros(E, dtype=i32, device="cuda")
    offs = torch.zeros(E + 1, dtype=i32, device="cuda")
    r2t = torch.zeros(mc, dtype=i32, device="cuda")
    tsr = torch.zeros((T, k), dtype=i32, device="cuda")
    am_t = torch.zeros(T, dtype=f32, device="cuda")
    am_r = torch.zeros(mc, dtype=f32, device="cuda")
    pws = torch.empty(M.permute_workspace_bytes(T, E), dtype=torch.uint8, device="cuda")
    xd = dev(x)
    M.moe_permute_amax(dev(lg), None, None, xd, T, E, k, d, ids, w, counts, offs, r2t, tsr, am_t, am_r, pws)
    xq = M.empty_quantized(mc, d)
    M.nvfp4_quantize_rows(xd, d, r2t, am_t, mc, xq["codes"], xq["sf"], xq["g"])
    hq = M.empty_quantized(mc, dff)
    f1ws = torch.empty(M.fc1_workspace_bytes(dff), dtype=torch.uint8, device="cuda")
    M.nvfp4_grouped_gemm_fc1_swiglu(xq["codes"], xq["sf"], xq["g"], offs, E, mc, d, dff, w1q["codes"],
                                    w1q["sf"], w1q["g"], hq["codes"], hq["sf"], hq["g"], None, None, f1ws)
    slots = torch.zeros((mc, d), dtype=torch.int16, device="cuda")
    out = torch.zeros((T, d), dtype=torch.int16, device="cuda")
    M.nvfp4_grouped_gemm_fc2_unpermute(hq["codes"], hq["sf"], hq["g"], offs, E, mc, dff, d, w2q["codes"],
                                       w2q["sf"], w2q["g"], r2t, tsr, w, T, k, slots, out, None)
    torch.cuda.synchronize()
    mp = int(host(offs)[-1])
    assert np.array_equal(host(xq["codes"])[:mp], r["x_codes"][:mp])
    assert np.array_equal(host(hq["codes"])[:mp], r["h_codes"][:mp])
    assert np.array_equal(host(out, np.uint16), r["out"])


def test_forward_deterministic(orc):
    lay = synth.layer("small")
    x, lg, W1, W2 = lay.x(), lay.logits(), lay.w1(), lay.w2()
    r1, w1q, w2q = gpu_forward(lay, x, lg, W1, W2)
    r2, _, _ = gpu_forward(lay, x, lg, w1q=w1q, w2q=w2q)
    for key in ["out", "row_to_token", "token_slot_row"]:
        assert np.array_equal(r1[key], r2[key]), key
    # the per-row buffers are written below offsets[E] only; the rest of the
    # workspace is whatever the allocation held
    mp = int(r1["offsets"][-1])
    for key in ["h_codes", "x_codes", "h_g", "x_g", "slots"]:
        assert np.array_equal(r1[key][:mp], r2[key][:mp]), key


def test_forward_flags_nonfinite_and_guards_memory(orc):
    import torch
    from gpu_util import dev, host
    lay = synth.layer("tiny")
    x, lg, W1, W2 = lay.x(), lay.logits(), lay.w1(), lay.w2()
    x = x.copy()
    lg = lg.copy()
    x[3, 7] = 0x7FC0     # NaN
    lg[5, 1] = np.inf
    r, w1q, w2q = gpu_forward(lay, x, lg, W1, W2)
    assert r["status"] & M.STATUS_NONFINITE_X and r["status"] & M.STATUS_NONFINITE_LOGITS
    # guard band after the output buffer
    T, d = lay.T, lay.d
    x, lg = lay.x(), lay.logits()
    G = 8192
    buf = torch.full((T * d + G,), 0x3C3C, dtype=torch.int16, device="cuda")
    ws = M.forward_workspace(T, lay.E, lay.k, d, lay.d_ff)
    wsg = torch.full((ws.numel() + G,), 0xEE, dtype=torch.uint8, device="cuda")
    M.moe_expert_forward(dev(x), dev(lg), T, lay.E, lay.k, d, lay.d_ff, w1q["codes"], w1q["sf"], w1q["g"],
                         w2q["codes"], w2q["sf"], w2q["g"], buf, wsg[:ws.numel()])
    torch.cuda.synchronize()
    assert np.all(host(buf)[T * d:] == 0x3C3C)
    assert np.all(host(wsg)[ws.numel():] == 0xEE)


def test_forward_empty_batch(orc):
    import torch
    lay = synth.layer("tiny")
    W = torch.zeros((lay.E, 2 * lay.d_ff, lay.d), dtype=torch.int16, device="cuda")
    W2 = torch.zeros((lay.E, lay.d, lay.d_ff), dtype=torch.int16, device="cuda")
    w1q, w2q = M.quantize_weights(W), M.quantize_weights(W2)
    M.moe_expert_forward(None, None, 0, lay.E, lay.k, lay.d, lay.d_ff, w1q["codes"], w1q["sf"], w1q["g"],
                         w2q["codes"], w2q["sf"], w2q["g"], None, None)


@pytest.mark.parametrize("name", ["qwen16k", "qwen64k"])
def test_full_size_sampled_tokens(orc, name):
    """The full Qwen-shaped workload in the launch configuration bench.py
    times; sampled tokens (first, last, and a spread) checked one by one."""
    import torch
    from gpu_util import dev
    lay = synth.layer(name)
    x, lg = lay.x(), lay.logits()
    W1, W2 = lay.w1(), lay.w2()
    r, _, _ = gpu_forward(lay, x, lg, W1, W2)
    assert r["status"] == 0
    ids, w = orc.route(lg, lay.k)
    perm = orc.permute(ids, lay.E)
    assert np.array_equal(r["topk_ids"], ids)
    for key in ["counts", "offsets", "token_slot_row"]:
        assert np.array_equal(r[key], perm[key]), key
    tok = orc.TokenOracle(W1, W2, lay.k)
    T = lay.T
    sample = sorted(set([0, 1, T // 3, T // 2, T - 2, T - 1] + list(np.random.default_rng(0).integers(0, T, 6))))
    got, exp, slots = [], [], []
    for t in sample:
        o = tok.token(x[t], lg[t])
        for j in range(lay.k):
            row = r["token_slot_row"][t, j]
            assert np.array_equal(r["x_codes"][row], o["x_codes"])
            assert r["x_g"][row] == o["x_g"]
        got.append(r["out"][t])
        exp.append(o["out"])
        slots.append(o["slots"])
    rel, mx, ratio = e2e_errors(np.stack(got), np.stack(exp), np.stack(slots))
    print("%s sampled %d tokens: rel-L2 %.3e max-abs %.3e (%.2f of the flip bound)" % (name, len(sample), rel, mx, ratio))
    assert rel <= E2E_REL_L2 and ratio <= 1.0


def test_forward_timed_equals_forward(orc):
    """moe_expert_forward_timed runs the same seven launches as
    moe_expert_forward (same output, bit for bit) and records the caller's
    eight events around them, in order."""
    import torch
    from gpu_util import dev, host
    lay = synth.layer("small")
    x, lg, W1, W2 = lay.x(), lay.logits(), lay.w1(), lay.w2()
    T, E, k, d, dff = lay.T, lay.E, lay.k, lay.d, lay.d_ff
    r, w1q, w2q = gpu_forward(lay, x, lg, W1, W2)
    out = torch.full((T, d), 0x5A5A, dtype=torch.int16, device="cuda")
    ws = M.forward_workspace(T, E, k, d, dff)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    M.moe_expert_forward_timed(dev(x), dev(lg), T, E, k, d, dff, w1q["codes"], w1q["sf"], w1q["g"], w2q["codes"],
                               w2q["sf"], w2q["g"], out, ws, st, None, ev)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(host(out, np.uint16), r["out"])
    times = [ev[0].elapsed_time(e) for e in ev]
    assert all(b >= a for a, b in zip(times, times[1:])) and times[-1] > 0
    # no events: refused before anything is enqueued
    assert M.lib().moe_expert_forward_timed(None, None, T, E, k, d, dff, None, None, None, None, None, None, None,
                                            None, 0, None, None, None) == M.MOE_ERR_POINTER
