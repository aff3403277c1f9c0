"""The C-ABI library loads without a GPU, exports every function its header
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes

import pytest

import nvfp4_w4a4_moe_top_gb300 as M


@pytest.fixture(scope="module")
def L():
    from nvfp4_w4a4_moe_top_gb300 import build
    build.build()
    return M.lib()


def test_exports_every_header_function(L):
    names = M.header_functions()
    assert len(names) == 26, names
    for n in names:
        assert hasattr(L, n), n
    for n in ["moe_nvfp4_quantize_weights", "moe_nvfp4_quantize_weights_per_expert", "moe_permute_amax", "nvfp4_quantize_rows",
              "nvfp4_grouped_gemm_fc1_swiglu", "nvfp4_grouped_gemm_fc2_unpermute", "moe_expert_forward",
              "moe_expert_forward_train", "moe_expert_backward", "moe_expert_backward_workspace_bytes",
              "moe_expert_forward_gather", "moe_expert_forward_timed", "moe_pipeline_device_bytes",
              "moe_pipeline_create",
              "moe_pipeline_submit", "moe_pipeline_synchronize", "moe_pipeline_destroy"]:
        assert n in names


def test_helpers_match_oracle(L, orc):
    assert M.abi_version() == 1
    for T, E, k in [(256, 8, 2), (4096, 32, 4), (65536, 128, 8), (1, 128, 8), (0, 8, 2), (3, 1, 1)]:
        assert M.m_cap(T, E, k) == orc.m_cap(T, E, k)
    for rows, K in [(128, 64), (1000, 2048), (1, 768)]:
        assert M.sf_bytes(rows, K) == orc.sf_bytes(rows, K)
    assert M.sf_bytes(10, 48) == 0
    assert M.status_string(-3) == "workspace too small"
    # h staging: two 128 x d_ff BF16 buffers per CTA, 256 CTAs at most
    # h staging (two 128 x d_ff BF16 buffers per CTA) + 16 deferred-SwiGLU slots of 16 B per epilogue thread
    assert M.fc1_workspace_bytes(768) == 256 * 2 * 128 * 768 * 2 + 256 * 512 * 16 * 16
    mc = M.m_cap(65536, 128, 8)
    assert M.backward_workspace_bytes(65536, 128, 8, 2048, 768) == mc * 2048 * 2 * 2 + mc * 1536 * 2 + mc * 2048 * 4
    assert M.backward_workspace_bytes(10, 4, 2, 200, 128) == 0


def test_workspace_layout_is_disjoint_and_aligned(L):
    for shape in [(256, 8, 2, 256, 128), (65536, 128, 8, 2048, 768), (1, 4, 4, 128, 128)]:
        lay = M.forward_workspace_layout(*shape)
        total = M.forward_workspace_bytes(*shape)
        offs = [lay[n] for n in M.WS_FIELDS]
        assert offs == sorted(offs) and all(o % 1024 == 0 for o in offs)
        assert offs[-1] < total
    T, E, k, d, dff = 65536, 128, 8, 2048, 768
    lay = M.forward_workspace_layout(T, E, k, d, dff)
    mc = M.m_cap(T, E, k)
    assert lay["x_sf"] - lay["x_codes"] >= mc * d // 2
    assert lay["chunk_hist"] - lay["slots"] >= M.m_cap(T, E, k) * d * 2


FAKE = ctypes.c_void_p(1 << 20)        # aligned, never dereferenced
MIS = ctypes.c_void_p((1 << 20) + 8)   # misaligned


def _fwd(L, T=256, E=8, k=2, d=256, dff=128, x=FAKE, ws=FAKE, ws_bytes=1 << 40, w=FAKE):
    return L.moe_expert_forward(x, FAKE, T, E, k, d, dff, w, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                ws, ws_bytes, None, None)


def test_forward_rejects_bad_arguments(L):
    assert _fwd(L, k=3, E=2) == M.MOE_ERR_SHAPE
    assert _fwd(L, d=200) == M.MOE_ERR_SHAPE
    assert _fwd(L, dff=64) == M.MOE_ERR_SHAPE
    assert _fwd(L, E=2000) == M.MOE_ERR_SHAPE
    assert _fwd(L, k=33, E=64) == M.MOE_ERR_SHAPE
    assert _fwd(L, T=-1) == M.MOE_ERR_SHAPE
    assert _fwd(L, x=None) == M.MOE_ERR_POINTER
    assert _fwd(L, x=MIS) == M.MOE_ERR_POINTER
    assert _fwd(L, w=None) == M.MOE_ERR_POINTER
    assert _fwd(L, ws_bytes=1024) == M.MOE_ERR_WORKSPACE
    # the gather-on-load forward validates identically
    g = [FAKE, FAKE, 256, 8, 2, 256, 128] + [FAKE] * 7
    assert L.moe_expert_forward_gather(*g, FAKE, 1024, None, None) == M.MOE_ERR_WORKSPACE
    assert L.moe_expert_forward_gather(*(g[:5] + [200] + g[6:]), FAKE, 1 << 40, None, None) == M.MOE_ERR_SHAPE
    assert L.moe_expert_forward_gather(*(g[:5] + [128] + g[6:]), FAKE, 1 << 40, None, None) == M.MOE_ERR_SHAPE


def test_entry_points_reject_bad_arguments(L):
    assert L.moe_nvfp4_quantize_weights(FAKE, 2, 100, 64, FAKE, FAKE, FAKE, None, None) == M.MOE_ERR_SHAPE
    assert L.moe_nvfp4_quantize_weights(FAKE, 2, 128, 48, FAKE, FAKE, FAKE, None, None) == M.MOE_ERR_SHAPE
    assert L.moe_nvfp4_quantize_weights(None, 2, 128, 64, FAKE, FAKE, FAKE, None, None) == M.MOE_ERR_POINTER
    # backward: shape, pointer and workspace checks before any CUDA call
    bw = [FAKE, FAKE, 256, 8, 2, 256, 128] + [FAKE] * 18 + [None, FAKE, FAKE]
    assert L.moe_expert_backward(*bw, 16, None, None) == M.MOE_ERR_WORKSPACE
    bad = list(bw)
    bad[5] = 200
    assert L.moe_expert_backward(*bad, 1 << 40, None, None) == M.MOE_ERR_SHAPE
    bad = list(bw)
    bad[7] = None  # W1
    assert L.moe_expert_backward(*bad, 1 << 40, None, None) == M.MOE_ERR_POINTER
    bad = list(bw)
    bad[19] = MIS  # h codes
    assert L.moe_expert_backward(*bad, 1 << 40, None, None) == M.MOE_ERR_POINTER
    ft = [FAKE, FAKE, 256, 8, 2, 256, 128] + [FAKE] * 7 + [FAKE, 1 << 40, None, FAKE, None, None]
    assert L.moe_expert_forward_train(*ft) == M.MOE_ERR_POINTER
    # pipeline: sizes and argument checks before any CUDA call
    ws = M.forward_workspace_bytes(256, 8, 2, 256, 128)
    up = lambda n: (n + 1023) // 1024 * 1024
    slot = up(256 * 256 * 2) * 2 + up(256 * 8 * 4)
    assert L.moe_pipeline_device_bytes(256, 8, 2, 256, 128, 3) == 3 * slot + up(ws)
    assert L.moe_pipeline_device_bytes(256, 8, 2, 256, 128, 5) == 0
    assert L.moe_pipeline_device_bytes(0, 8, 2, 256, 128, 2) == 0
    h = ctypes.c_void_p()
    assert L.moe_pipeline_create(256, 8, 2, 256, 128, 2, FAKE, 16, ctypes.byref(h)) == M.MOE_ERR_WORKSPACE
    assert L.moe_pipeline_create(256, 8, 2, 256, 128, 2, MIS, 1 << 40, ctypes.byref(h)) == M.MOE_ERR_POINTER
    assert L.moe_pipeline_create(256, 8, 2, 200, 128, 2, FAKE, 1 << 40, ctypes.byref(h)) == M.MOE_ERR_SHAPE
    assert L.moe_pipeline_create(256, 8, 2, 256, 128, 2, FAKE, 1 << 40, None) == M.MOE_ERR_POINTER
    assert L.moe_pipeline_submit(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == M.MOE_ERR_POINTER
    assert L.moe_pipeline_destroy(None) == M.MOE_OK
    qe = L.moe_nvfp4_quantize_weights_per_expert
    assert qe(FAKE, 2, 100, 64, FAKE, FAKE, FAKE, FAKE, None, None) == M.MOE_ERR_SHAPE
    assert qe(FAKE, 0, 128, 64, FAKE, FAKE, FAKE, FAKE, None, None) == M.MOE_ERR_SHAPE
    assert qe(FAKE, 2, 128, 64, FAKE, FAKE, FAKE, None, None, None) == M.MOE_ERR_POINTER
    assert qe(FAKE, 2, 128, 64, FAKE, FAKE, FAKE, MIS, None, None) == M.MOE_ERR_POINTER
    assert L.nvfp4_quantize_rows(FAKE, 4, 100, None, None, 4, FAKE, FAKE, FAKE, None, None) == M.MOE_ERR_SHAPE
    assert L.nvfp4_quantize_rows(FAKE, 4, 64, None, None, 5, FAKE, FAKE, FAKE, None, None) == M.MOE_ERR_SHAPE
    assert L.nvfp4_quantize_rows(FAKE, 4, 64, MIS, None, 4, FAKE, FAKE, FAKE, None, None) == M.MOE_ERR_POINTER
    args = [FAKE, None, None, FAKE, 256, 8, 2, 256] + [FAKE] * 8
    assert L.moe_permute_amax(*args, FAKE, 4, None, None) == M.MOE_ERR_WORKSPACE
    bad = list(args)
    bad[6] = 9
    assert L.moe_permute_amax(*bad, FAKE, 1 << 30, None, None) == M.MOE_ERR_SHAPE
    bad = list(args)
    bad[0] = None
    assert L.moe_permute_amax(*bad, FAKE, 1 << 30, None, None) == M.MOE_ERR_POINTER
    # the no-allocation variant rejects shapes whose histograms exceed its
    # fixed scratch array before any CUDA call
    na = [FAKE, None, None, FAKE, 600000, 128, 2, 256] + [FAKE] * 8 + [None, None]
    assert L.moe_permute_amax_noalloc(*na) == M.MOE_ERR_WORKSPACE
    na[5] = 2000
    assert L.moe_permute_amax_noalloc(*na) == M.MOE_ERR_SHAPE
    fc1 = [FAKE] * 4 + [8, 1024, 256, 128] + [FAKE] * 8 + [FAKE]
    assert L.nvfp4_grouped_gemm_fc1_swiglu(*fc1, 16, None, None) == M.MOE_ERR_WORKSPACE
    fc1b = list(fc1)
    fc1b[5] = 1000
    assert L.nvfp4_grouped_gemm_fc1_swiglu(*fc1b, 1 << 40, None, None) == M.MOE_ERR_SHAPE
    fc2 = [FAKE] * 4 + [8, 1024, 128, 256] + [FAKE] * 6 + [256, 2] + [FAKE, FAKE, None, None, None]
    bad = list(fc2)
    bad[15] = 9
    assert L.nvfp4_grouped_gemm_fc2_unpermute(*bad) == M.MOE_ERR_SHAPE
    bad = list(fc2)
    bad[0] = MIS
    assert L.nvfp4_grouped_gemm_fc2_unpermute(*bad) == M.MOE_ERR_POINTER
