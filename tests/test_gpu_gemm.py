"""Parity of the tcgen05 grouped GEMMs with the oracle.

Inputs come from the oracle (routing, permutation, quantised activations and
weights).  Checks, per the specification's tolerance rules:
  FC1: pre-cast FP32 outputs (dbg_u) within rel-L2 1e-5 of the oracle's
       sequential-FP32 GEMM (every row); h bit-exact with the oracle SwiGLU
       of the GPU's u; h codes / scales / g bit-exact with the oracle's
       quantisation of the GPU's h.
  FC2: pre-weighting expert outputs y2 (dbg_y) within rel-L2 1e-5 and BF16
       max-abs 2e-3 of the oracle; the slots (z rows, slot (t, j) at row
       token_slot_row[t][j]) bit-exact with the oracle's weighting of the
       GPU's y2; out bit-exact with the oracle's reduce of the GPU's slots.
The debug outputs select a separate instantiation of each GEMM kernel; the
production instantiation (no debug pointers, the one the forward runs) is
tied to it bit for bit on the same inputs, including a 2048-token slice of
the Qwen-shaped layer (d = 2048, d_ff = 768, E = 128, top-8, Zipf-skewed
routing with empty experts: CTA pairs, eight resident A slices, six chunks).
"""
import functools
import numpy as np
import pytest

import nvfp4_w4a4_moe_top_gb300 as M
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from nvfp4_w4a4_moe_top_gb300 import build
    build.build()


@functools.lru_cache(maxsize=4)
def _case(name, T):
    import oracle as orc
    return make_case(orc, layer_of(name), T)


def make_case(orc, lay, T=None):
    x, lg, W1, W2 = lay.x(), lay.logits(), lay.w1(), lay.w2()
    if T is not None:
        x, lg = x[:T], lg[:T]
    T = x.shape[0]
    ids, w = orc.route(lg, lay.k)
    perm = orc.permute(ids, lay.E)
    am = orc.amax_rows(x)
    mc = perm["m_cap"]
    xq = orc.quantize_rows(x, perm["row_to_token"], am, mc)
    return dict(T=T, x=x, ids=ids, w=w, perm=perm, xq=xq, mc=mc,
                w1q=orc.quantize_weights(W1), w2q=orc.quantize_weights(W2))


def run_fc1(lay, c, debug=True):
    """FC1 on the case's inputs; debug=False runs the production
    instantiation (no debug outputs)."""
    import torch
    from gpu_util import dev, host
    mc, d, dff, E = c["mc"], lay.d, lay.d_ff, lay.E
    hq = M.empty_quantized(mc, dff)
    dbg_u = torch.full((mc, 2 * dff), float("nan"), dtype=torch.float32, device="cuda") if debug else None
    dbg_h = torch.zeros((mc, dff), dtype=torch.int16, device="cuda") if debug else None
    ws = torch.empty(M.fc1_workspace_bytes(dff), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    xc, xs, xg = c["xq"]
    w1c, w1s, w1g = c["w1q"]
    M.nvfp4_grouped_gemm_fc1_swiglu(dev(xc), dev(xs), dev(xg), dev(c["perm"]["offsets"]), E, mc, d, dff,
                                    dev(w1c), dev(w1s), dev(w1g), hq["codes"], hq["sf"], hq["g"], dbg_u, dbg_h,
                                    ws, st)
    torch.cuda.synchronize()
    r = dict(status=int(st.item()), h_codes=host(hq["codes"]), h_sf=host(hq["sf"]), h_g=host(hq["g"]))
    if debug:
        r.update(u=host(dbg_u), h=host(dbg_h, np.uint16))
    return r


CASES = [("tiny", None), ("small", None), ("custom_d128", None), ("custom_skew", None), ("custom_many_units", None),
         ("qwen_slice", 2048)]


def layer_of(name):
    if name == "custom_d128":
        return synth.custom(T=300, d=128, E=3, k=2, d_ff=256, seed=4)
    if name == "custom_many_units":
        # K = 128 in both GEMMs: one k-step per item, hundreds of units per
        # launch, so the producers run many units ahead of the MMAs
        return synth.custom(T=6000, d=128, E=4, k=2, d_ff=128, seed=6)
    if name == "custom_pair_skew":
        # d and d_ff multiples of 256, empty experts and experts with an odd
        # tile count (the last CTA-pair unit of such an expert has one tile)
        return synth.custom(T=900, d=512, E=10, k=3, d_ff=512, seed=9, logits="bias", bias_std=2.5,
                            n_forced_empty=3)
    if name == "custom_pair_3stage":
        # d = 2048 with d_ff = 1024: four 22 KB pair stages no longer fit beside
        # the resident A and the weight scales, so the pair plan takes three
        # (scale buffers then released by their own barrier)
        return synth.custom(T=320, d=2048, E=4, k=2, d_ff=1024, seed=12)
    if name == "custom_skew":
        return synth.custom(T=700, d=384, E=16, k=3, d_ff=384, seed=5, logits="bias", bias_std=3.0,
                            n_forced_empty=5)
    if name == "qwen_slice":
        return synth.layer("qwen16k")
    return synth.layer(name)


@pytest.mark.parametrize("name,T", CASES)
def test_fc1_parity(orc, name, T):
    from gpu_util import rel_l2
    lay = layer_of(name)
    c = _case(name, T)
    g = run_fc1(lay, c)
    assert g["status"] == 0
    mp = c["perm"]["m_pad"]
    xc, xs, xg = c["xq"]
    y1 = orc.grouped_gemm(xc, xs, xg, c["perm"]["offsets"], *c["w1q"], lay.d, 2 * lay.d_ff)
    assert rel_l2(g["u"][:mp], y1[:mp]) <= 1e-5
    # per-row: every row within 1e-5 relative (rows with a nonzero reference)
    nr = np.linalg.norm(y1[:mp], axis=1)
    rows = nr > 0
    assert np.all(np.linalg.norm(g["u"][:mp] - y1[:mp], axis=1)[rows] <= 1e-5 * nr[rows])
    # SwiGLU of the GPU's own FC1 output: bit-exact (h = BF16(silu(g) up),
    # one rounding, on both sides)
    _, h_ref = orc.swiglu(g["u"][:mp], lay.d_ff)
    assert np.array_equal(g["h"][:mp], h_ref)
    # requantisation of the GPU's h: bit-exact
    hc, hs, hg = orc.quantize_rows(g["h"][:mp])
    assert np.array_equal(g["h_codes"][:mp], hc)
    assert np.array_equal(g["h_g"][:mp].view(np.uint32), hg.view(np.uint32))
    assert np.array_equal(orc.unswizzle_sf(g["h_sf"], mp, lay.d_ff), orc.unswizzle_sf(hs, mp, lay.d_ff))
    # pad rows come out as zero rows
    pad = c["perm"]["row_to_token"][:mp] < 0
    assert not g["h_codes"][:mp][pad].any() and not g["h_g"][:mp][pad].any()


def run_fc2(lay, c, hq, debug=True):
    import torch
    from gpu_util import dev, host
    mc, d, dff, E, T, k = c["mc"], lay.d, lay.d_ff, lay.E, c["T"], lay.k
    slots = torch.zeros((mc, d), dtype=torch.int16, device="cuda")
    out = torch.zeros((T, d), dtype=torch.int16, device="cuda")
    dbg_y = torch.full((mc, d), float("nan"), dtype=torch.float32, device="cuda") if debug else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    w2c, w2s, w2g = c["w2q"]
    M.nvfp4_grouped_gemm_fc2_unpermute(dev(hq[0]), dev(hq[1]), dev(hq[2]), dev(c["perm"]["offsets"]), E, mc, dff,
                                       d, dev(w2c), dev(w2s), dev(w2g), dev(c["perm"]["row_to_token"]),
                                       dev(c["perm"]["token_slot_row"]), dev(c["w"]), T, k, slots, out, dbg_y, st)
    torch.cuda.synchronize()
    r = dict(status=int(st.item()), slots=host(slots, np.uint16), out=host(out, np.uint16))
    if debug:
        r["y"] = host(dbg_y)
    return r


@pytest.mark.parametrize("name,T", CASES)
def test_fc2_parity(orc, name, T):
    from gpu_util import rel_l2, f32_of_bf16
    lay = layer_of(name)
    c = _case(name, T)
    mp, mc = c["perm"]["m_pad"], c["mc"]
    # FC2 operand: the oracle's own FC1 -> SwiGLU -> requantisation
    xc, xs, xg = c["xq"]
    y1 = orc.grouped_gemm(xc, xs, xg, c["perm"]["offsets"], *c["w1q"], lay.d, 2 * lay.d_ff)
    _, h = orc.swiglu(y1, lay.d_ff)
    hq = orc.quantize_rows(h)
    g = run_fc2(lay, c, hq)
    assert g["status"] == 0
    y2 = orc.grouped_gemm(hq[0], hq[1], hq[2], c["perm"]["offsets"], *c["w2q"], lay.d_ff, lay.d)
    real = c["perm"]["row_to_token"][:mp] >= 0
    gy, ey = g["y"][:mp][real], y2[:mp][real]
    assert rel_l2(gy, ey) <= 1e-5
    from helpers import torch_bf16
    assert np.abs(f32_of_bf16(torch_bf16(gy)) - f32_of_bf16(torch_bf16(ey))).max() <= 2e-3
    # router-weighted BF16 scatter of the GPU's y2, and the reduce: bit-exact
    y_full = np.zeros_like(y2)
    y_full[:mp] = g["y"][:mp]
    slots_ref = orc.combine(y_full, c["perm"], c["w"], c["T"], lay.k, lay.d)
    slots = g["slots"][c["perm"]["token_slot_row"]]  # [T][k][d]
    assert np.array_equal(slots, slots_ref)
    assert np.array_equal(g["out"], orc.reduce(slots))
    # pad rows of the z rows are written as zeros
    assert not g["slots"][:mp][~real].any()


@pytest.mark.parametrize("name", ["small", "custom_skew", "custom_pair_skew", "custom_pair_3stage"])
def test_fc1_cta_pairs_equal_single(orc, name, monkeypatch):
    """FC1 on CTA pairs (cta_group::2 MMAs over 256-row units, the default
    where the pair plan fits) and on single CTAs produce the same bits: the
    same K order per output element, only the tile's rows split over two
    SMs.  custom_skew has empty experts and experts with an odd tile count,
    whose last pair unit leaves rank 1 without a tile of its own."""
    lay = layer_of(name)
    c = make_case(orc, lay)
    mp = c["perm"]["m_pad"]
    g2 = run_fc1(lay, c)
    monkeypatch.setenv("MOE_FC1_CTA_PAIRS", "0")
    g1 = run_fc1(lay, c)
    assert g1["status"] == 0 and g2["status"] == 0
    assert np.array_equal(g2["u"][:mp].view(np.uint32), g1["u"][:mp].view(np.uint32))
    assert np.array_equal(g2["h"][:mp], g1["h"][:mp])
    assert np.array_equal(g2["h_codes"][:mp], g1["h_codes"][:mp])
    assert np.array_equal(g2["h_g"][:mp].view(np.uint32), g1["h_g"][:mp].view(np.uint32))
    assert np.array_equal(orc.unswizzle_sf(g2["h_sf"], mp, lay.d_ff), orc.unswizzle_sf(g1["h_sf"], mp, lay.d_ff))


@pytest.mark.parametrize("name,T", [("small", None), ("custom_skew", None), ("custom_pair_skew", None),
                                    ("qwen_slice", 2048)])
def test_production_kernels_equal_debug(orc, name, T):
    """The production instantiations (no debug pointers: the kernels the
    forward and bench.py run) give the same h codes, block scales and g, and
    the same slots and output, bit for bit, as the debug instantiations that
    the oracle checks above; so they meet the same parity."""
    lay = layer_of(name)
    c = _case(name, T)
    mp = c["perm"]["m_pad"]
    gd = run_fc1(lay, c, debug=True)
    gp = run_fc1(lay, c, debug=False)
    assert gd["status"] == 0 and gp["status"] == 0
    assert np.array_equal(gp["h_codes"][:mp], gd["h_codes"][:mp])
    assert np.array_equal(gp["h_g"][:mp].view(np.uint32), gd["h_g"][:mp].view(np.uint32))
    assert np.array_equal(orc.unswizzle_sf(gp["h_sf"], mp, lay.d_ff), orc.unswizzle_sf(gd["h_sf"], mp, lay.d_ff))
    # and the production h is the oracle's requantisation of the (debug) h
    hc, hs, hg = orc.quantize_rows(gd["h"][:mp])
    assert np.array_equal(gp["h_codes"][:mp], hc)
    # FC2 on the GPU's quantised h, both instantiations
    hq = (gp["h_codes"], gp["h_sf"], gp["h_g"])
    fd = run_fc2(lay, c, hq, debug=True)
    fp = run_fc2(lay, c, hq, debug=False)
    assert fd["status"] == 0 and fp["status"] == 0
    assert np.array_equal(fp["slots"], fd["slots"])
    assert np.array_equal(fp["out"], fd["out"])
