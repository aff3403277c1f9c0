"""Bit-exact parity of routing, permutation, padding, expert offsets and
per-token amax (moe_permute_amax) with the oracle; router weights within
FP32 rounding."""
import numpy as np
import pytest

import nvfp4_w4a4_moe_top_gb300 as M
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from nvfp4_w4a4_moe_top_gb300 import build
    build.build()


def run_permute(T, E, k, d, logits=None, x=None, ext_ids=None, ext_w=None):
    import torch
    from gpu_util import dev, host
    mc = M.m_cap(T, E, k)
    i32, f32 = torch.int32, torch.float32
    o = dict(topk_ids=torch.zeros((T, k), dtype=i32, device="cuda"),
             topk_w=torch.zeros((T, k), dtype=f32, device="cuda"),
             counts=torch.zeros(E, dtype=i32, device="cuda"),
             offsets=torch.zeros(E + 1, dtype=i32, device="cuda"),
             row_to_token=torch.full((max(mc, 1),), 77, dtype=i32, device="cuda"),
             token_slot_row=torch.zeros((T, k), dtype=i32, device="cuda"),
             amax_tok=torch.zeros(max(T, 1), dtype=f32, device="cuda"),
             amax_row=torch.full((max(mc, 1),), 5.0, dtype=f32, device="cuda"))
    ws = torch.empty(max(M.permute_workspace_bytes(T, E), 16), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=i32, device="cuda")
    M.moe_permute_amax(None if logits is None else dev(logits), None if ext_ids is None else dev(ext_ids),
                       None if ext_w is None else dev(ext_w), None if x is None else dev(x), T, E, k, d,
                       o["topk_ids"], o["topk_w"], o["counts"], o["offsets"], o["row_to_token"],
                       o["token_slot_row"], o["amax_tok"], o["amax_row"], ws, st)
    torch.cuda.synchronize()
    r = {n: host(t) for n, t in o.items()}
    r["row_to_token"] = r["row_to_token"][:mc]
    r["amax_row"] = r["amax_row"][:mc]
    r["status"] = int(st.item())
    return r


def check(orc, r, ids, w, x, E):
    perm = orc.permute(ids, E)
    assert r["status"] == 0
    assert np.array_equal(r["topk_ids"], ids)
    assert np.allclose(r["topk_w"], w, rtol=1e-6, atol=0)
    for key in ["counts", "offsets", "row_to_token", "token_slot_row"]:
        assert np.array_equal(r[key], perm[key]), key
    if x is not None:
        am = orc.amax_rows(x)
        assert np.array_equal(r["amax_tok"][:len(am)].view(np.uint32), am.view(np.uint32))
        exp_row = np.where(perm["row_to_token"] >= 0, am[np.maximum(perm["row_to_token"], 0)], 0).astype(np.float32)
        assert np.array_equal(r["amax_row"].view(np.uint32), exp_row.view(np.uint32))
    return perm


@pytest.mark.parametrize("name", ["tiny", "small", "qwen16k"])
def test_permute_amax_configs(orc, name):
    lay = synth.layer(name)
    lg, x = lay.logits(), lay.x()
    r = run_permute(lay.T, lay.E, lay.k, lay.d, logits=lg, x=x)
    ids, w = orc.route(lg, lay.k)
    perm = check(orc, r, ids, w, x, lay.E)
    if name == "small":
        assert (perm["counts"] == 0).sum() >= 2


@pytest.mark.parametrize("T,E,k", [(1, 4, 4), (300, 1, 1), (517, 5, 3), (1000, 256, 8), (70, 1024, 32),
                                   (2049, 64, 6)])
def test_permute_ragged_shapes(orc, T, E, k):
    rng = np.random.default_rng(T + E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[:, 0] += 3.0                                         # one hot expert
    lg[: T // 3, :] = np.round(lg[: T // 3, :])             # many ties
    x = synth.to_bf16_bits(rng.standard_normal((T, 128)).astype(np.float32))
    r = run_permute(T, E, k, 128, logits=lg, x=x)
    ids, w = orc.route(lg, k)
    check(orc, r, ids, w, x, E)


def test_routing_replay(orc):
    rng = np.random.default_rng(3)
    T, E, k = 700, 16, 4
    ids = np.sort(np.stack([rng.choice(E, k, replace=False) for _ in range(T)]), axis=1).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    r = run_permute(T, E, k, 0, ext_ids=ids, ext_w=w)
    assert r["status"] == 0
    assert np.array_equal(r["topk_ids"], ids) and np.array_equal(r["topk_w"], w)
    perm = orc.permute(ids, E)
    for key in ["counts", "offsets", "row_to_token", "token_slot_row"]:
        assert np.array_equal(r[key], perm[key]), key
    bad = ids.copy()
    bad[5, 1] = bad[5, 0]
    bad[9, 2] = 99
    assert run_permute(T, E, k, 0, ext_ids=bad, ext_w=w)["status"] & M.STATUS_BAD_ROUTING


def test_nonfinite_logits_flagged(orc):
    lg = np.zeros((10, 8), np.float32)
    lg[4, 2] = np.nan
    r = run_permute(10, 8, 2, 0, logits=lg)
    assert r["status"] & M.STATUS_NONFINITE_LOGITS


def test_empty_batch(orc):
    r = run_permute(0, 8, 2, 128, logits=np.zeros((0, 8), np.float32), x=np.zeros((0, 128), np.uint16))
    assert not r["counts"].any() and not r["offsets"].any()
