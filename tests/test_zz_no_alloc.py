"""moe_permute_amax_noalloc, the entry point for callers that cannot allocate
device memory (a plugin of a runtime that owns all device memory, a serving
loop that must not call cudaMalloc on its hot path): it keeps its histogram
scratch in a fixed array inside the library.

Called through the C ABI twice in a row on different inputs, its results
must equal, bit for bit, those of moe_permute_amax given a workspace of its
own (same kernels, so the same bits), which the oracle parity tests pin.
This file is collected last on purpose; it must also pass on its own in a
fresh process."""
import numpy as np
import pytest

import nvfp4_w4a4_moe_top_gb300 as M
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from nvfp4_w4a4_moe_top_gb300 import build
    build.build()


def _outputs(T, E, k):
    import torch
    mc = M.m_cap(T, E, k)
    i32, f32 = torch.int32, torch.float32
    return dict(topk_ids=torch.full((T, k), -3, dtype=i32, device="cuda"),
                topk_w=torch.full((T, k), -3.0, dtype=f32, device="cuda"),
                counts=torch.full((E,), -3, dtype=i32, device="cuda"),
                offsets=torch.full((E + 1,), -3, dtype=i32, device="cuda"),
                row_to_token=torch.full((mc,), 77, dtype=i32, device="cuda"),
                token_slot_row=torch.full((T, k), -3, dtype=i32, device="cuda"),
                amax_tok=torch.full((T,), -3.0, dtype=f32, device="cuda"),
                amax_row=torch.full((mc,), 5.0, dtype=f32, device="cuda"),
                status=torch.zeros(1, dtype=i32, device="cuda"))


def _host(o):
    return {n: t.cpu().numpy() for n, t in o.items()}


def _run_pair(T, E, k, d, lg, x):
    import torch
    from gpu_util import dev
    lg_d, x_d = dev(lg), dev(x)
    ref = _outputs(T, E, k)
    ws = torch.empty(max(M.permute_workspace_bytes(T, E), 16), dtype=torch.uint8, device="cuda")
    M.moe_permute_amax(lg_d, None, None, x_d, T, E, k, d, ref["topk_ids"], ref["topk_w"], ref["counts"],
                       ref["offsets"], ref["row_to_token"], ref["token_slot_row"], ref["amax_tok"],
                       ref["amax_row"], ws, ref["status"])
    got = _outputs(T, E, k)
    M.moe_permute_amax_noalloc(lg_d, None, None, x_d, T, E, k, d, got["topk_ids"], got["topk_w"],
                               got["counts"], got["offsets"], got["row_to_token"], got["token_slot_row"],
                               got["amax_tok"], got["amax_row"], got["status"])
    torch.cuda.synchronize()
    return _host(ref), _host(got)


def _assert_same(ref, got):
    assert int(ref["status"][0]) == 0 and int(got["status"][0]) == 0
    for n in ref:
        a, b = ref[n], got[n]
        if a.dtype == np.float32:
            a, b = a.view(np.uint32), b.view(np.uint32)
        assert np.array_equal(a, b), n


def test_noalloc_matches_workspace_entry_point_twice():
    # first call: the small layer (ragged groups, two empty experts); second
    # call right after on a different shape whose histogram is larger, so
    # stale contents of the shared array from the first call would show
    lay = synth.layer("small")
    ref, got = _run_pair(lay.T, lay.E, lay.k, lay.d, lay.logits(), lay.x())
    _assert_same(ref, got)
    assert (ref["counts"] == 0).sum() >= 2

    rng = np.random.default_rng(2049)
    T, E, k, d = 2049, 64, 6, 128
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[:, 3] += 2.5
    x = synth.to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    ref2, got2 = _run_pair(T, E, k, d, lg, x)
    _assert_same(ref2, got2)


def test_noalloc_rejects_shapes_beyond_its_array():
    import torch
    from gpu_util import dev
    T, E, k, d = 600000, 128, 1, 128                 # 9375 chunks x 128 experts x 4 B > 4 MiB
    assert M.permute_workspace_bytes(T, E) > (1 << 22)
    one = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(M.MoeError) as ei:
        M.moe_permute_amax_noalloc(one, None, None, one, T, E, k, d, one, one, one, one, one, one, one, one)
    assert ei.value.code == M.MOE_ERR_WORKSPACE
