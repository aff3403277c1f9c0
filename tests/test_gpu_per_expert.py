"""Parity of the per-expert weight outer scale recipe ("miniTE CUTLASS"
column of the Technical Report's section 4.3 table) with the oracle.

moe_nvfp4_quantize_weights_per_expert: codes, block scales, the replicated
g and amax_e bit-exact with oracle.quantize_weights_per_expert, on small and
ragged shapes, an all-zero expert, a single expert, rows spanning several
decades, replays of a CUDA graph that captured the call, and sampled
experts of the full Qwen-shaped W1 and W2.  The forward
on per-expert weights (same GEMM kernels, per-expert g in the epilogue)
against the oracle forward on the oracle's per-expert weights.
"""
import numpy as np
import pytest

import nvfp4_w4a4_moe_top_gb300 as M
import synth
from helpers import bf16, f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from nvfp4_w4a4_moe_top_gb300 import build
    build.build()


def gpu_per_expert(W):
    import torch
    from gpu_util import dev, host
    q = M.quantize_weights_per_expert(dev(W))
    torch.cuda.synchronize()
    return host(q["codes"]), host(q["sf"]), host(q["g"]), host(q["amax_e"])


def check_equal(orc, W, got, experts=None):
    """got = the GPU's (codes, sf, g, amax_e) of all of W; the oracle runs on
    the listed experts only (each expert's result depends on its own tensor)."""
    E, N, K = W.shape
    codes, sf, g, am = got
    logical = orc.unswizzle_sf(sf, E * N, K)
    for e in (range(E) if experts is None else experts):
        ec, es, eg = orc.quantize_weights_per_expert(W[e][None])
        assert np.array_equal(codes[e], ec[0]), e
        assert np.array_equal(g[e].view(np.uint32), eg[0].view(np.uint32)), e
        assert np.array_equal(logical[e * N:(e + 1) * N], orc.unswizzle_sf(es, N, K)), e
        assert am[e] == np.float32(np.abs(f32(W[e])).max()), e


def wide_range_weights(E, N, K, seed):
    rng = np.random.default_rng(seed)
    scale = 10.0 ** rng.uniform(-4.0, 0.5, (E, N, 1)) * 0.02
    return bf16((rng.standard_normal((E, N, K)) * scale).astype(np.float32))


def test_small_layer_weights_bitexact(orc):
    lay = synth.layer("small")
    for W in (np.stack([lay.w1_expert(e) for e in range(4)]), np.stack([lay.w2_expert(e) for e in range(4)])):
        check_equal(orc, W, gpu_per_expert(W))


@pytest.mark.parametrize("E,N,K", [(3, 128, 192), (1, 256, 64), (5, 384, 4096), (2, 128, 1024), (13, 128, 256),
                                   (17, 256, 128)])
def test_wide_range_and_zero_expert(orc, E, N, K):
    W = wide_range_weights(E, N, K, seed=E * 7 + K)
    if E > 1:
        W[1] = 0  # an all-zero expert: g = 0, every scale and code +0
    got = gpu_per_expert(W)
    check_equal(orc, W, got)
    if E > 1:
        assert got[3][1] == 0 and not got[2][1].any() and not got[0][1].any()


def test_extreme_expert_scales(orc):
    """Experts whose outer scale leaves [2^-87, 2^111] (maxima near 1e-30 and
    1e37): encoded by the fix-up pass with the E2M1 division's row factor,
    bit-exact all the same, beside an ordinary expert."""
    rng = np.random.default_rng(21)
    W = np.stack([rng.standard_normal((256, 512)) * s for s in (1e-30, 0.02, 1e37)]).astype(np.float32)
    W = bf16(W)
    check_equal(orc, W, gpu_per_expert(W))


def test_per_expert_differs_from_per_row(orc):
    """The two recipes really differ on the GPU: same codes as the per-row
    call only where a row's amax equals its expert's."""
    import torch
    from gpu_util import dev, host
    W = wide_range_weights(2, 128, 256, seed=3)
    ce, se, ge, am = gpu_per_expert(W)
    qr = M.quantize_weights(dev(W))
    torch.cuda.synchronize()
    gr = host(qr["g"])
    row_amax = np.abs(f32(W)).max(axis=2)
    top = row_amax == am[:, None]
    assert np.array_equal(ge[top].view(np.uint32), gr[top].view(np.uint32))
    assert np.all(ge[~top] > gr[~top])


def test_nonfinite_weight_sets_status(orc):
    import torch
    from gpu_util import dev, host
    W = np.zeros((2, 128, 64), np.float32)
    W[1, 7, 7] = np.nan
    W[0, 3, 3] = 0.5
    q = M.empty_quantized(256, 64)
    am = torch.empty(2, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_nvfp4_quantize_weights_per_expert(dev(bf16(W).reshape(2, 128, 64)), q["codes"], q["sf"], q["g"], am, st)
    torch.cuda.synchronize()
    assert int(st.item()) & M.STATUS_NONFINITE_WEIGHT
    a = host(am)
    assert a[0] == np.float32(0.5) and a[1] == 0.0  # NaN does not win the maximum


def test_replays_in_a_cuda_graph(orc):
    """Captured on a stream in a CUDA graph (the memset of amax_e and both
    launches), then replayed on new weights copied into the captured buffer:
    every replay equals the oracle, so the maxima restart from zero on each
    replay."""
    import torch
    from gpu_util import dev, host
    E, N, K = 11, 128, 256
    W = dev(wide_range_weights(E, N, K, seed=5))
    q = M.empty_quantized(E * N, K)
    am = torch.empty(E, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()

    def call():
        M.moe_nvfp4_quantize_weights_per_expert(W, q["codes"], q["sf"], q["g"], am, st)

    with torch.cuda.stream(s):  # first call outside the capture: device checks
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for seed in [6, 7]:
        Wn = wide_range_weights(E, N, K, seed=seed)
        Wn[seed % E] = 0
        W.copy_(dev(Wn))
        g.replay()
        torch.cuda.synchronize()
        got = (host(q["codes"]).reshape(E, N, K // 2), host(q["sf"]), host(q["g"]).reshape(E, N), host(am))
        check_equal(orc, Wn, got)
    assert int(st.item()) == 0


@pytest.mark.parametrize("which", ["w1", "w2"])
def test_full_size_sampled_experts(orc, which):
    """The Qwen-shaped expert weights (128 experts; W1 1536 x 2048, W2
    2048 x 768), all quantised in one call, sampled experts checked."""
    lay = synth.layer("qwen16k")
    get = lay.w1_expert if which == "w1" else lay.w2_expert
    W = np.stack([get(e) for e in range(lay.E)])
    got = gpu_per_expert(W)
    check_equal(orc, W, got, experts=[0, 1, 37, 64, 126, 127])


@pytest.mark.parametrize("name", ["tiny", "small", "ragged"])
def test_forward_with_per_expert_weights(orc, name):
    import torch
    from gpu_util import dev, host, f32_of_bf16, rel_l2
    if name == "ragged":
        lay = synth.custom(T=999, d=384, E=12, k=3, d_ff=256, seed=11, logits="bias", bias_std=2.0,
                           n_forced_empty=3)
    else:
        lay = synth.layer(name)
    x, lg, W1, W2 = lay.x(), lay.logits(), lay.w1(), lay.w2()
    T, E, k, d, dff = lay.T, lay.E, lay.k, lay.d, lay.d_ff
    w1q, w2q = M.quantize_weights_per_expert(dev(W1)), M.quantize_weights_per_expert(dev(W2))
    out = torch.empty((T, d), dtype=torch.int16, device="cuda")
    ws = M.forward_workspace(T, E, k, d, dff)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_expert_forward(dev(x), dev(lg), T, E, k, d, dff, w1q["codes"], w1q["sf"], w1q["g"], w2q["codes"],
                         w2q["sf"], w2q["g"], out, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.moe_forward(x, lg, orc.quantize_weights_per_expert(W1), orc.quantize_weights_per_expert(W2), k, dff)
    v = M.forward_views(ws, T, E, k, d, dff)
    mp = ref["perm"]["m_pad"]
    assert np.array_equal(host(v["x_codes"])[:mp], ref["x_codes"][:mp])
    row_diff = np.any(host(v["h_codes"])[:mp] != ref["h_codes"][:mp], axis=1)
    from test_gpu_forward import E2E_REL_L2, H_ROWS_DIFFERING, e2e_errors
    rel, mx, ratio = e2e_errors(host(out, np.uint16), ref["out"], ref["slots"])
    print("%s per-expert weights: e2e rel-L2 %.3e max-abs %.3e (%.2f of the flip bound), h-code rows differing %.5f"
          % (name, rel, mx, ratio, row_diff.mean()))
    # the same end-to-end tolerance as the per-row forward
    assert row_diff.mean() <= H_ROWS_DIFFERING
    assert rel <= E2E_REL_L2 and ratio <= 1.0
