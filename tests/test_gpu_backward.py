"""Parity of the straight-through BF16 backward (moe_expert_forward_train +
moe_expert_backward) with the oracle.  The backward recomputes the
forward's expert outputs y2 (FC2 again on the saved FP4 operands); the
oracle gets the forward's y2 from the modular FC2's debug output.

Stage-wise, the oracle fed the GPU's own saved forward values (u, h, y2 and
the routing, which are bit-exact with the oracle's forward):
  dy2 and the permuted x: bit-exact;
  du: equal up to rare BF16 flips (dh accumulates in a different order on
      the tensor cores), rel-L2 <= 1e-4;
  dW2 (no BF16 step after dy2): rel-L2 <= 1e-5;
  dw, dlogits: rel-L2 <= 1e-4;
  dx, dW1 (through du): rel-L2 <= 3e-4 -- the du flips dominate, about
      sqrt(flip fraction) * 2^-8 (measured 1e-5 .. 1e-4).
End to end against the fully independent oracle (its own forward, then its
own backward): rel-L2 <= 1e-3 on dx, dW1, dW2 (the tolerance stated for the
forward-plus-backward workload).  At the Qwen-shaped 64k-token layer the
same call is checked on sampled tokens (dx) and whole experts (dW1, dW2).
"""
import numpy as np
import pytest

import nvfp4_w4a4_moe_top_gb300 as M
import synth
from helpers import f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from nvfp4_w4a4_moe_top_gb300 import build
    build.build()


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    n = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (n if n > 0 else 1.0))


def gpu_train_step(lay, x, lg, W1, W2, dY):
    """Forward with saved values, then the backward, on the GPU."""
    import torch
    from gpu_util import dev, host
    T, E, k, d, F = x.shape[0], lay.E, lay.k, lay.d, lay.d_ff
    W1d, W2d = dev(W1), dev(W2)
    w1q, w2q = M.quantize_weights(W1d), M.quantize_weights(W2d)
    mc = M.m_cap(T, E, k)
    out = torch.empty((T, d), dtype=torch.int16, device="cuda")
    ws = M.forward_workspace(T, E, k, d, F)
    su = torch.full((mc, 2 * F), 0x7FC0, dtype=torch.int16, device="cuda")
    sh = torch.full((mc, F), 0x7FC0, dtype=torch.int16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_expert_forward_train(dev(x), dev(lg), T, E, k, d, F, w1q["codes"], w1q["sf"], w1q["g"], w2q["codes"],
                               w2q["sf"], w2q["g"], out, ws, su, sh, st)
    v = M.forward_views(ws, T, E, k, d, F)
    # the forward's FP32 expert outputs, for the oracle only: the modular FC2
    # on the same requantised h (its debug output), into scratch buffers
    sy = torch.full((mc, d), float("nan"), dtype=torch.float32, device="cuda")
    M.nvfp4_grouped_gemm_fc2_unpermute(v["h_codes"], v["h_sf"], v["h_g"], v["offsets"], E, mc, F, d, w2q["codes"],
                                       w2q["sf"], w2q["g"], v["row_to_token"], v["token_slot_row"], v["topk_w"], T,
                                       k, torch.empty((mc, d), dtype=torch.int16, device="cuda"),
                                       torch.empty((T, d), dtype=torch.int16, device="cuda"), sy)
    dx = torch.full((T, d), float("nan"), dtype=torch.float32, device="cuda")
    dW1 = torch.full((E, 2 * F, d), float("nan"), dtype=torch.float32, device="cuda")
    dW2 = torch.full((E, d, F), float("nan"), dtype=torch.float32, device="cuda")
    dl = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    dw = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    bws = torch.empty(M.backward_workspace_bytes(T, E, k, d, F), dtype=torch.uint8, device="cuda")
    M.moe_expert_backward(dev(dY), dev(x), T, E, k, d, F, W1d, W2d, w2q["codes"], w2q["sf"], w2q["g"], v["topk_ids"],
                          v["topk_w"], v["offsets"], v["row_to_token"], v["token_slot_row"], su, sh, v["h_codes"],
                          v["h_sf"], v["h_g"], dx, dW1, dW2, dl, dw, bws, st)
    torch.cuda.synchronize()
    mp = int(host(v["offsets"])[-1])
    r = {n: host(t) for n, t in v.items() if n in ("topk_ids", "topk_w", "offsets", "row_to_token",
                                                    "token_slot_row", "counts")}
    r.update(status=int(st.item()), out=host(out, np.uint16), u=host(su, np.uint16), h=host(sh, np.uint16),
             y2=host(sy), dx=host(dx), dW1=host(dW1), dW2=host(dW2), dlogits=host(dl), dw=host(dw), m_pad=mp)
    L = bws.numel()
    o_dy2, o_xp, o_du = 0, (mc * d * 2 + 1023) // 1024 * 1024, 0
    o_du = o_xp + (mc * d * 2 + 1023) // 1024 * 1024
    r["dy2"] = host(bws[o_dy2:o_dy2 + mp * d * 2].view(torch.int16).view(mp, d), np.uint16)
    r["xp"] = host(bws[o_xp:o_xp + mp * d * 2].view(torch.int16).view(mp, d), np.uint16)
    r["du"] = host(bws[o_du:o_du + mp * 2 * F * 2].view(torch.int16).view(mp, 2 * F), np.uint16)
    assert o_du + mc * 2 * F * 2 <= L
    return r


def fwd_from_gpu(r, T):
    """The oracle's forward-result dict built from the GPU's saved values."""
    mp = r["m_pad"]
    perm = dict(offsets=r["offsets"], row_to_token=r["row_to_token"], token_slot_row=r["token_slot_row"],
                m_pad=mp, counts=r["counts"])
    return dict(ids=r["topk_ids"], w=r["topk_w"], perm=perm, u=r["u"][:mp], h=r["h"][:mp], y2=r["y2"][:mp])


def layer_of(name):
    if name == "ragged":
        return synth.custom(T=999, d=384, E=12, k=3, d_ff=256, seed=11, logits="bias", bias_std=2.0,
                            n_forced_empty=3)
    if name == "k1":
        return synth.custom(T=130, d=256, E=4, k=1, d_ff=128, seed=2)
    if name == "ragged_pairs":
        # d a multiple of 256, so the FC2 recomputation runs on CTA pairs (three
        # rings, scale buffers on their own ring), with empty experts and odd
        # tile counts (ghost tiles)
        return synth.custom(T=1500, d=512, E=12, k=3, d_ff=256, seed=13, logits="bias", bias_std=2.0,
                            n_forced_empty=3)
    return synth.layer(name)


@pytest.mark.parametrize("name", ["tiny", "small", "ragged", "k1", "ragged_pairs"])
def test_backward_against_oracle(orc, name):
    lay = layer_of(name)
    x, lg, W1, W2, dY = lay.x(), lay.logits(), lay.w1(), lay.w2(), lay.grad_out()
    r = gpu_train_step(lay, x, lg, W1, W2, dY)
    assert r["status"] == 0
    mp = r["m_pad"]
    # saved forward values are the forward's own (routing bit-exact)
    ref = orc.moe_forward(x, lg, orc.quantize_weights(W1), orc.quantize_weights(W2), lay.k, lay.d_ff)
    assert np.array_equal(r["topk_ids"], ref["ids"])
    assert np.array_equal(r["offsets"], ref["perm"]["offsets"])
    real = r["row_to_token"][:mp] >= 0
    # (y2 cascades the forward's rare h-code flips: the forward's own
    # end-to-end tolerance)
    assert rel(r["y2"][:mp][real], ref["y2"][:mp][real]) <= 2e-3
    # stage-wise: the oracle backward of the GPU's saved values
    g = orc.moe_backward(dY, x, W1, W2, fwd_from_gpu(r, lay.T))
    assert np.array_equal(r["dy2"], g["dy2"])
    assert np.array_equal(r["xp"], orc.gather_x_rows(x, r["row_to_token"][:mp]))
    diff = r["du"].astype(np.int32) - g["du"].astype(np.int32)
    flips = diff != 0
    print("%s: du flips %d of %d" % (name, int(flips.sum()), flips.size))
    assert flips.mean() <= 1e-3
    # a flip is one BF16 ulp of a rounding decision, or a sign where dh
    # cancels to about zero: negligible in norm
    assert rel(f32(r["du"]), f32(g["du"])) <= 1e-4
    errs = {key: rel(r[key], g[key]) for key in ["dx", "dW1", "dW2", "dw", "dlogits"]}
    print("%s stage-wise rel-L2: %s" % (name, ", ".join("%s %.2e" % kv for kv in errs.items())))
    assert errs["dW2"] <= 1e-5
    for key in ["dw", "dlogits"]:
        assert errs[key] <= 1e-4, key
    for key in ["dx", "dW1"]:
        assert errs[key] <= 3e-4, key
    # end to end against the independent oracle
    gi = orc.moe_backward(dY, x, W1, W2, ref)
    e2e = {key: rel(r[key], gi[key]) for key in ["dx", "dW1", "dW2"]}
    print("%s end-to-end rel-L2: %s" % (name, ", ".join("%s %.2e" % kv for kv in e2e.items())))
    for key in ["dx", "dW1", "dW2"]:
        assert e2e[key] <= 1e-3, key


@pytest.mark.parametrize("name", ["small", "tiny"])
def test_backward_cta_pairs_equal_single(orc, name, monkeypatch):
    """The backward GEMMs on CTA pairs (where N, and for the weight
    gradients Mo, are multiples of 256) and on single CTAs: every gradient
    bit for bit."""
    lay = layer_of(name)
    x, lg, W1, W2, dY = lay.x(), lay.logits(), lay.w1(), lay.w2(), lay.grad_out()
    r2 = gpu_train_step(lay, x, lg, W1, W2, dY)
    monkeypatch.setenv("MOE_BWD_CTA_PAIRS", "0")
    r1 = gpu_train_step(lay, x, lg, W1, W2, dY)
    assert r1["status"] == 0 and r2["status"] == 0
    for key in ("du", "dx", "dW1", "dW2", "dw", "dlogits"):
        assert np.array_equal(r1[key].view(np.uint8), r2[key].view(np.uint8)), key


@pytest.mark.parametrize("name", ["small", "tiny", "ragged_pairs"])
def test_backward_fc2_pairs_equal_single(orc, name, monkeypatch):
    """The backward's FC2 recomputation on CTA pairs and on single CTAs: dy2
    and every gradient that flows from it bit for bit; dw (a dot product
    over d, summed in four column parts on pairs and two on single CTAs)
    and the logit gradient within FP32 reassociation."""
    lay = layer_of(name)
    x, lg, W1, W2, dY = lay.x(), lay.logits(), lay.w1(), lay.w2(), lay.grad_out()
    r2 = gpu_train_step(lay, x, lg, W1, W2, dY)
    monkeypatch.setenv("MOE_FC2_CTA_PAIRS", "0")
    r1 = gpu_train_step(lay, x, lg, W1, W2, dY)
    assert r1["status"] == 0 and r2["status"] == 0
    for key in ("dy2", "du", "dx", "dW1", "dW2"):
        assert np.array_equal(r1[key].view(np.uint8), r2[key].view(np.uint8)), key
    for key in ("dw", "dlogits"):
        assert rel(r2[key], r1[key]) <= 1e-6, key


@pytest.mark.parametrize("name", ["small", "ragged"])
def test_backward_side_stream_equals_one_stream(orc, name, monkeypatch):
    """The permuted-row copy on the second stream (beside the GEMMs) and on
    the caller's stream: every gradient bit for bit."""
    lay = layer_of(name)
    x, lg, W1, W2, dY = lay.x(), lay.logits(), lay.w1(), lay.w2(), lay.grad_out()
    r2 = gpu_train_step(lay, x, lg, W1, W2, dY)
    monkeypatch.setenv("MOE_BWD_SIDE_STREAM", "0")
    r1 = gpu_train_step(lay, x, lg, W1, W2, dY)
    assert r1["status"] == 0 and r2["status"] == 0
    for key in ("xp", "du", "dx", "dW1", "dW2", "dw", "dlogits"):
        assert np.array_equal(r1[key].view(np.uint8), r2[key].view(np.uint8)), key


def test_empty_experts_get_zero_weight_gradients(orc):
    lay = layer_of("ragged")
    x, lg, W1, W2, dY = lay.x(), lay.logits(), lay.w1(), lay.w2(), lay.grad_out()
    r = gpu_train_step(lay, x, lg, W1, W2, dY)
    empty = np.where(np.diff(r["offsets"]) == 0)[0]
    assert len(empty) >= 3
    assert not r["dW1"][empty].any() and not r["dW2"][empty].any()
    assert np.all(np.isfinite(r["dW1"])) and np.all(np.isfinite(r["dW2"])) and np.all(np.isfinite(r["dx"]))


def test_backward_is_deterministic(orc):
    lay = layer_of("tiny")
    x, lg, W1, W2, dY = lay.x(), lay.logits(), lay.w1(), lay.w2(), lay.grad_out()
    a = gpu_train_step(lay, x, lg, W1, W2, dY)
    b = gpu_train_step(lay, x, lg, W1, W2, dY)
    for key in ["dx", "dW1", "dW2", "dw", "dlogits", "du"]:
        assert np.array_equal(a[key], b[key]), key


def test_full_size_sampled(orc):
    """The 64k-token Qwen-shaped layer (forward plus backward workload): dx of
    sampled tokens and the weight gradients of two whole experts against the
    oracle run on the GPU's saved values of exactly those rows."""
    lay = synth.layer("qwen64k")
    x, lg, dY = lay.x(), lay.logits(), lay.grad_out()
    W1, W2 = lay.w1(), lay.w2()
    r = gpu_train_step(lay, x, lg, W1, W2, dY)
    assert r["status"] == 0
    w, tsr, offs, r2t = r["topk_w"], r["token_slot_row"], r["offsets"], r["row_to_token"]
    # the expert of each row
    expert_of_row = np.searchsorted(offs, np.arange(r["m_pad"]), side="right") - 1
    T = lay.T
    sample = sorted(set([0, 1, T // 2, T - 1] + list(np.random.default_rng(1).integers(0, T, 4))))
    got, exp = [], []
    for t in sample:
        acc = np.zeros(lay.d, np.float64)
        for j in range(lay.k):
            row = int(tsr[t, j])
            e = int(expert_of_row[row])
            dy2 = orc.bwd_dy2(dY[t:t + 1], w[t:t + 1, j:j + 1], np.zeros((1, 1), np.int32), 1)
            assert np.array_equal(dy2[0], r["dy2"][row])
            _, dxr, _, _ = orc.bwd_expert(dy2, r["u"][row:row + 1], r["h"][row:row + 1], x[t:t + 1], W1[e], W2[e])
            acc += dxr[0]
        got.append(r["dx"][t])
        exp.append(acc)
    e_dx = rel(np.stack(got), np.stack(exp))
    errs = []
    for e in [0, lay.E - 1]:
        a, b = int(offs[e]), int(offs[e + 1])
        _, _, dW1e, dW2e = orc.bwd_expert(r["dy2"][a:b], r["u"][a:b], r["h"][a:b],
                                          orc.gather_x_rows(x, r2t[a:b]), W1[e], W2[e])
        errs.append((rel(r["dW1"][e], dW1e), rel(r["dW2"][e], dW2e)))
    print("qwen64k: dx sampled rel-L2 %.2e; dW1/dW2 experts %s" % (e_dx, errs))
    assert e_dx <= 3e-4
    for a1, a2 in errs:
        assert a1 <= 3e-4 and a2 <= 1e-5


def test_training_forward_output_equals_the_forward(orc):
    """moe_expert_forward_train returns what moe_expert_forward returns, bit
    for bit (the saves do not change the arithmetic)."""
    import torch
    from gpu_util import dev, host
    lay = layer_of("ragged")
    x, lg, W1, W2, dY = lay.x(), lay.logits(), lay.w1(), lay.w2(), lay.grad_out()
    r = gpu_train_step(lay, x, lg, W1, W2, dY)
    T, E, k, d, F = lay.T, lay.E, lay.k, lay.d, lay.d_ff
    w1q, w2q = M.quantize_weights(dev(W1)), M.quantize_weights(dev(W2))
    out = torch.empty((T, d), dtype=torch.int16, device="cuda")
    M.moe_expert_forward(dev(x), dev(lg), T, E, k, d, F, w1q["codes"], w1q["sf"], w1q["g"], w2q["codes"], w2q["sf"],
                         w2q["g"], out, M.forward_workspace(T, E, k, d, F))
    torch.cuda.synchronize()
    assert np.array_equal(r["out"], host(out, np.uint16))


def test_backward_of_an_empty_batch_zeroes_the_weight_gradients(orc):
    import torch
    lay = layer_of("tiny")
    E, k, d, F = lay.E, lay.k, lay.d, lay.d_ff
    W1 = torch.ones((E, 2 * F, d), dtype=torch.int16, device="cuda")
    W2 = torch.ones((E, d, F), dtype=torch.int16, device="cuda")
    dW1 = torch.full((E, 2 * F, d), float("nan"), dtype=torch.float32, device="cuda")
    dW2 = torch.full((E, d, F), float("nan"), dtype=torch.float32, device="cuda")
    M.moe_expert_backward(None, None, 0, E, k, d, F, W1, W2, None, None, None, None, None, None, None, None, None,
                          None, None, None, None, None, dW1, dW2, None, None, None)
    torch.cuda.synchronize()
    assert not dW1.any() and not dW2.any()
