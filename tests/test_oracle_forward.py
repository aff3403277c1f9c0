"""End-to-end properties of the oracle's expert forward and of the seeded
input recipe."""
import numpy as np
import pytest

import synth
from helpers import f32, bf16


@pytest.fixture(scope="module")
def tiny(orc):
    lay = synth.layer("tiny")
    x, lg, W1, W2 = lay.x(), lay.logits(), lay.w1(), lay.w2()
    w1q, w2q = orc.quantize_weights(W1), orc.quantize_weights(W2)
    res = orc.moe_forward(x, lg, w1q, w2q, lay.k, lay.d_ff)
    return lay, x, lg, W1, W2, w1q, w2q, res


def test_token_oracle_equals_full_forward(orc, tiny):
    lay, x, lg, W1, W2, w1q, w2q, res = tiny
    tok = orc.TokenOracle(W1, W2, lay.k)
    for t in [0, 1, 77, 255]:
        r = tok.token(x[t], lg[t])
        assert np.array_equal(r["ids"], res["ids"][t])
        assert np.array_equal(r["out"], res["out"][t])
        for j in range(lay.k):
            row = res["perm"]["token_slot_row"][t, j]
            assert np.array_equal(r["h"][j], res["h"][row])
            assert np.array_equal(r["y2"][j], res["y2"][row])


def test_results_do_not_depend_on_thread_count(orc, tiny):
    """The oracle's parallel loops give every output to one thread, summed in
    a fixed order: one thread and all threads give the same bits."""
    lay, x, lg, W1, W2, w1q, w2q, res = tiny
    n0 = orc.num_threads()
    orc.set_num_threads(1)
    try:
        assert orc.num_threads() == 1 or n0 == 1
        one = orc.moe_forward(x, lg, w1q, w2q, lay.k, lay.d_ff)
    finally:
        orc.set_num_threads(n0)
    assert orc.num_threads() == n0
    for key in ("out", "y2", "h", "slots"):
        assert np.array_equal(one[key], res[key]), key


def test_context_swap_invariance_end_to_end(orc, tiny):
    """Replacing and reordering the other tokens leaves a token's codes and
    output bitwise unchanged (per-token scales, RHT and stochastic rounding
    off: the context-swap check of the AI summary's methodology)."""
    lay, x, lg, W1, W2, w1q, w2q, res = tiny
    target = 17
    rng = np.random.default_rng(99)
    x2 = bf16(rng.standard_normal(x.shape) * 7)
    lg2 = rng.standard_normal(lg.shape).astype(np.float32)
    perm = rng.permutation(lay.T)
    x2, lg2 = x2[perm], lg2[perm]
    pos = int(np.nonzero(perm == 0)[0][0])
    x2[pos], lg2[pos] = x[target], lg[target]
    res2 = orc.moe_forward(x2, lg2, w1q, w2q, lay.k, lay.d_ff)
    assert np.array_equal(res2["out"][pos], res["out"][target])
    for j in range(lay.k):
        r1 = res["perm"]["token_slot_row"][target, j]
        r2 = res2["perm"]["token_slot_row"][pos, j]
        assert np.array_equal(res2["x_codes"][r2], res["x_codes"][r1])
        assert np.array_equal(res2["h_codes"][r2], res["h_codes"][r1])


def test_pad_rows_are_zero(orc, tiny):
    lay, x, lg, W1, W2, w1q, w2q, res = tiny
    r2t = res["perm"]["row_to_token"]
    pad = r2t < 0
    assert pad.any()
    assert not res["x_codes"][pad].any() and not res["x_g"][pad].any()
    assert not res["h_codes"][pad[:len(res["h_codes"])]].any()
    assert np.all(res["amax_row"][pad] == 0)


def test_quantized_forward_tracks_fp64_reference(orc, tiny):
    """NVFP4 W4A4 output against an unquantised FP64 SwiGLU FFN on the same
    BF16 inputs: relative L2 error of the order of the format's own error."""
    lay, x, lg, W1, W2, w1q, w2q, res = tiny
    X = f32(x).astype(np.float64)
    ref = np.zeros_like(X)
    for t in range(lay.T):
        for j in range(lay.k):
            e, w = res["ids"][t, j], res["w"][t, j]
            u = f32(W1[e]).astype(np.float64) @ X[t]
            g, up = u[:lay.d_ff], u[lay.d_ff:]
            h = g / (1 + np.exp(-g)) * up
            ref[t] += w * (f32(W2[e]).astype(np.float64) @ h)
    out = f32(res["out"]).astype(np.float64)
    rel = np.linalg.norm(out - ref) / np.linalg.norm(ref)
    assert 0.03 < rel < 0.3, rel


def test_k1_single_expert(orc):
    lay = synth.custom(T=40, d=128, E=1, k=1, d_ff=128, seed=3)
    x, lg, W1, W2 = lay.x(), lay.logits(), lay.w1(), lay.w2()
    res = orc.moe_forward(x, lg, orc.quantize_weights(W1), orc.quantize_weights(W2), 1, 128)
    assert np.all(res["w"] == 1.0)
    # k = 1 and w = 1: the output is the BF16 cast of the expert output
    assert np.array_equal(res["out"], res["slots"][:, 0])


def test_synth_is_deterministic_and_blockwise(orc):
    a, b = synth.layer("tiny", seed=5), synth.layer("tiny", seed=5)
    assert np.array_equal(a.x(), b.x()) and np.array_equal(a.logits(), b.logits())
    assert np.array_equal(a.w1_expert(3), b.w1()[3])
    assert not np.array_equal(a.x(), synth.layer("tiny", seed=6).x())
    lay = synth.custom(T=2500, d=64, E=4, k=2, d_ff=64, seed=1)
    x = lay.x()
    assert np.array_equal(lay.x_rows([0, 1023, 1024, 2499]), x[[0, 1023, 1024, 2499]])
    assert np.array_equal(lay.logits_rows([5, 2048]), lay.logits()[[5, 2048]])


def test_small_recipe_has_empty_experts(orc):
    lay = synth.layer("small")
    ids, _ = orc.route(lay.logits(), lay.k)
    counts = np.bincount(ids.ravel(), minlength=lay.E)
    assert (counts == 0).sum() >= 2
    assert counts.max() > 3 * counts[counts > 0].min()       # skewed groups


def test_qwen16k_recipe_is_zipf_skewed(orc):
    lay = synth.layer("qwen16k")
    lg = np.concatenate([lay.logits_block(b) for b in range(4)])   # 4096 tokens
    ids, _ = orc.route(lg, lay.k)
    counts = np.sort(np.bincount(ids.ravel(), minlength=lay.E))[::-1]
    assert counts[0] > 5 * np.median(counts)
