"""Gather-on-load FC1 (moe_expert_forward_gather): each token quantised once,
FC1 fetching its A rows by row_to_token with TMA tile::gather4.

The result must equal moe_expert_forward bit for bit (same arithmetic, only
the data movement differs): output, routing, permutation, scales, g, h codes
and slots; the token-ordered codes equal the oracle's per-token quantisation
and the extra row T is zero.  Covered: ragged groups, empty experts, k = 1,
one expert, every expert selected, and the full 64k-token layer."""
import numpy as np
import pytest

import nvfp4_w4a4_moe_top_gb300 as M
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from nvfp4_w4a4_moe_top_gb300 import build
    build.build()


def run_both(lay, x, lg, W1, W2):
    import torch
    from gpu_util import dev, host
    T, E, k, d, F = x.shape[0], lay.E, lay.k, lay.d, lay.d_ff
    w1q, w2q = M.quantize_weights(dev(W1)), M.quantize_weights(dev(W2))
    xd, lgd = dev(x), dev(lg)
    res = []
    for fn in (M.moe_expert_forward, M.moe_expert_forward_gather):
        out = torch.full((T, d), 0x5A5A, dtype=torch.int16, device="cuda")
        ws = torch.full((M.forward_workspace_bytes(T, E, k, d, F),), 0xA5, dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        fn(xd, lgd, T, E, k, d, F, w1q["codes"], w1q["sf"], w1q["g"], w2q["codes"], w2q["sf"], w2q["g"], out, ws, st)
        torch.cuda.synchronize()
        v = M.forward_views(ws, T, E, k, d, F)
        r = {n: host(t) for n, t in v.items() if hasattr(t, "detach")}
        r["out"] = host(out, np.uint16)
        r["status"] = int(st.item())
        res.append(r)
    return res


def layer_of(name):
    if name == "ragged":
        return synth.custom(T=999, d=384, E=12, k=3, d_ff=256, seed=11, logits="bias", bias_std=2.0,
                            n_forced_empty=3)
    if name == "k1":
        return synth.custom(T=130, d=256, E=4, k=1, d_ff=128, seed=2)
    if name == "single_expert":
        return synth.custom(T=200, d=256, E=1, k=1, d_ff=128, seed=3)
    if name == "all_experts":
        return synth.custom(T=64, d=256, E=6, k=6, d_ff=256, seed=8)
    if name == "wide":  # K = 4096: A streams through the stages instead of staying resident
        return synth.custom(T=300, d=4096, E=4, k=2, d_ff=256, seed=12)
    return synth.layer(name)


def check(orc, lay, x, base, gat, full_oracle=True):
    assert base["status"] == 0 and gat["status"] == 0
    assert np.array_equal(gat["out"], base["out"])
    mp = int(base["offsets"][-1])
    for key in ["topk_ids", "topk_w", "token_slot_row", "counts", "offsets", "row_to_token", "amax_tok"]:
        assert np.array_equal(gat[key], base[key]), key
    assert np.array_equal(gat["x_g"][:mp], base["x_g"][:mp])
    assert np.array_equal(orc.unswizzle_sf(gat["x_sf"], mp, lay.d), orc.unswizzle_sf(base["x_sf"], mp, lay.d))
    assert np.array_equal(gat["h_codes"][:mp], base["h_codes"][:mp])
    assert np.array_equal(gat["h_g"][:mp], base["h_g"][:mp])
    T = x.shape[0]
    tok = gat["x_codes"][:T + 1]
    assert not tok[T].any()
    # the token-ordered codes are the per-row copies of the row-ordered path
    r2t = base["row_to_token"][:mp]
    real = r2t >= 0
    assert np.array_equal(tok[r2t[real]], base["x_codes"][:mp][real])
    if full_oracle:
        c, _, _ = orc.quantize_rows(x)
        assert np.array_equal(tok[:T], c)


@pytest.mark.parametrize("name", ["tiny", "small", "ragged", "k1", "single_expert", "all_experts", "wide"])
def test_gather_equals_row_copies(orc, name):
    lay = layer_of(name)
    x, lg, W1, W2 = lay.x(), lay.logits(), lay.w1(), lay.w2()
    base, gat = run_both(lay, x, lg, W1, W2)
    check(orc, lay, x, base, gat)


def test_gather_full_size():
    """The 64k-token Qwen-shaped layer in bench.py's launch configuration."""
    import oracle as orc
    lay = synth.layer("qwen64k")
    x, lg, W1, W2 = lay.x(), lay.logits(), lay.w1(), lay.w2()
    base, gat = run_both(lay, x, lg, W1, W2)
    check(orc, lay, x, base, gat, full_oracle=False)
    # sampled tokens of the token-ordered codes against the oracle
    T = x.shape[0]
    for t in [0, 1, T // 2, T - 1]:
        c, _, _ = orc.quantize_rows(x[t:t + 1])
        assert np.array_equal(gat["x_codes"][t], c[0])
