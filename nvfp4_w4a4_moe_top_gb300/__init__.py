"""Python binding of libmoe_nvfp4.so: the native NVFP4 W4A4 MoE expert
forward on one GB300 (sm_103a).

Argument marshalling only: every function passes torch tensors as device
pointers, the current CUDA stream, and raises ``MoeError`` on a negative
return code.  Every step of the computation runs in the library's CUDA
kernels; there is no CPU path.  The library must have been built
(``nvfp4_w4a4_moe_top_gb300.build.build()``); importing a missing library
raises.

Tensor conventions (see include/moe_nvfp4.h): bf16 data may be passed as
torch.bfloat16 or 16-bit integer tensors; all tensors are contiguous, on the
current CUDA device, 16-byte aligned.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe_nvfp4.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "moe_nvfp4.h")

MOE_OK, MOE_ERR_POINTER, MOE_ERR_SHAPE, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_DEVICE = 0, -1, -2, -3, -4, -5
STATUS_NONFINITE_X, STATUS_NONFINITE_LOGITS, STATUS_NONFINITE_WEIGHT = 0x1, 0x2, 0x4
STATUS_BAD_ROUTING, STATUS_TIMEOUT = 0x8, 0x10

WS_FIELDS = ["topk_ids", "topk_w", "token_slot_row", "counts", "offsets", "row_to_token",
             "amax_tok", "x_codes", "x_sf", "x_g", "h_codes", "h_sf", "h_g", "slots",
             "chunk_hist", "fc1_staging"]


class MoeError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__("%s failed: %d (%s)" % (fn, code, status_string(code)))


P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_SIGS = {
    "moe_abi_version": (I32, []),
    "moe_status_string": (ctypes.c_char_p, [I32]),
    "moe_m_cap": (I64, [I32, I32, I32]),
    "nvfp4_sf_bytes": (SZ, [I64, I32]),
    "moe_permute_workspace_bytes": (SZ, [I32, I32]),
    "nvfp4_fc1_workspace_bytes": (SZ, [I32]),
    "moe_expert_forward_workspace_bytes": (SZ, [I32, I32, I32, I32, I32]),
    "moe_expert_forward_workspace_layout": (I32, [I32, I32, I32, I32, I32, P]),
    "moe_nvfp4_quantize_weights": (I32, [P, I32, I32, I32, P, P, P, P, P]),
    "moe_nvfp4_quantize_weights_per_expert": (I32, [P, I32, I32, I32, P, P, P, P, P, P]),
    "moe_permute_amax": (I32, [P, P, P, P, I32, I32, I32, I32, P, P, P, P, P, P, P, P, P, SZ, P, P]),
    "moe_permute_amax_noalloc": (I32, [P, P, P, P, I32, I32, I32, I32, P, P, P, P, P, P, P, P, P, P]),
    "nvfp4_quantize_rows": (I32, [P, I32, I32, P, P, I32, P, P, P, P, P]),
    "nvfp4_grouped_gemm_fc1_swiglu": (I32, [P, P, P, P, I32, I64, I32, I32, P, P, P, P, P, P, P, P, P, SZ, P, P]),
    "nvfp4_grouped_gemm_fc2_unpermute": (I32, [P, P, P, P, I32, I64, I32, I32, P, P, P, P, P, P, I32, I32, P, P, P, P, P]),
    "moe_expert_forward": (I32, [P, P, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, P, SZ, P, P]),
    "moe_pipeline_device_bytes": (SZ, [I32, I32, I32, I32, I32, I32]),
    "moe_pipeline_create": (I32, [I32, I32, I32, I32, I32, I32, P, SZ, P]),
    "moe_pipeline_submit": (I32, [P, P, P, P, P, P, P, P, P, P, P]),
    "moe_pipeline_synchronize": (I32, [P]),
    "moe_pipeline_destroy": (I32, [P]),
    "moe_expert_forward_timed": (I32, [P, P, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, P, SZ, P, P, P]),
    "moe_expert_forward_gather": (I32, [P, P, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, P, SZ, P, P]),
    "moe_expert_forward_train": (I32, [P, P, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, P, SZ, P, P, P, P]),
    "moe_expert_backward_workspace_bytes": (SZ, [I32, I32, I32, I32, I32]),
    "moe_expert_backward": (I32, [P, P, I32, I32, I32, I32, I32] + [P] * 21 + [SZ, P, P]),
}

_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libmoe_nvfp4.so is not built: run nvfp4_w4a4_moe_top_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def header_functions():
    """Names of the functions include/moe_nvfp4.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z][a-z0-9_]*)\s*\(", src)) - {"defined"})


# --------------------------------------------------------------------------
def status_string(code):
    return lib().moe_status_string(int(code)).decode()


def abi_version():
    return lib().moe_abi_version()


def m_cap(T, E, k):
    return int(lib().moe_m_cap(T, E, k))


def sf_bytes(rows, K):
    return int(lib().nvfp4_sf_bytes(rows, K))


def permute_workspace_bytes(T, E):
    return int(lib().moe_permute_workspace_bytes(T, E))


def fc1_workspace_bytes(d_ff):
    return int(lib().nvfp4_fc1_workspace_bytes(d_ff))


def forward_workspace_bytes(T, E, k, d, d_ff):
    return int(lib().moe_expert_forward_workspace_bytes(T, E, k, d, d_ff))


def forward_workspace_layout(T, E, k, d, d_ff):
    arr = (ctypes.c_size_t * 16)()
    _check("moe_expert_forward_workspace_layout",
           lib().moe_expert_forward_workspace_layout(T, E, k, d, d_ff, ctypes.cast(arr, P)))
    return dict(zip(WS_FIELDS, list(arr)))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, rc):
    if rc != MOE_OK:
        raise MoeError(fn, rc)


# --------------------------------------------------------------------------
# entry points (same names and argument order as the C functions)
# --------------------------------------------------------------------------
def moe_nvfp4_quantize_weights(W, codes, sf, g, status=None, stream=None):
    E, N, K = W.shape
    _check("moe_nvfp4_quantize_weights",
           lib().moe_nvfp4_quantize_weights(_p(W), E, N, K, _p(codes), _p(sf), _p(g), _p(status), _s(stream)))


def moe_nvfp4_quantize_weights_per_expert(W, codes, sf, g, amax_e, status=None, stream=None):
    E, N, K = W.shape
    _check("moe_nvfp4_quantize_weights_per_expert", lib().moe_nvfp4_quantize_weights_per_expert(
        _p(W), E, N, K, _p(codes), _p(sf), _p(g), _p(amax_e), _p(status), _s(stream)))


def moe_permute_amax(logits, ext_ids, ext_w, x, T, E, k, d, topk_ids, topk_w, counts, offsets,
                     row_to_token, token_slot_row, amax_tok, amax_row, ws, status=None, stream=None):
    _check("moe_permute_amax", lib().moe_permute_amax(
        _p(logits), _p(ext_ids), _p(ext_w), _p(x), T, E, k, d, _p(topk_ids), _p(topk_w), _p(counts),
        _p(offsets), _p(row_to_token), _p(token_slot_row), _p(amax_tok), _p(amax_row), _p(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _p(status), _s(stream)))


def moe_permute_amax_noalloc(logits, ext_ids, ext_w, x, T, E, k, d, topk_ids, topk_w, counts, offsets,
                             row_to_token, token_slot_row, amax_tok, amax_row, status=None, stream=None):
    """moe_permute_amax with the library's own fixed scratch array instead of
    a workspace: for callers that cannot allocate device memory.  Calls that
    overlap on the GPU race on that array; see include/moe_nvfp4.h."""
    _check("moe_permute_amax_noalloc", lib().moe_permute_amax_noalloc(
        _p(logits), _p(ext_ids), _p(ext_w), _p(x), T, E, k, d, _p(topk_ids), _p(topk_w), _p(counts),
        _p(offsets), _p(row_to_token), _p(token_slot_row), _p(amax_tok), _p(amax_row), _p(status),
        _s(stream)))


def nvfp4_quantize_rows(src, K, row_map, amax, dst_rows, codes, sf, g, status=None, stream=None):
    src_rows = src.numel() // K
    _check("nvfp4_quantize_rows", lib().nvfp4_quantize_rows(
        _p(src), src_rows, K, _p(row_map), _p(amax), dst_rows, _p(codes), _p(sf), _p(g), _p(status),
        _s(stream)))


def nvfp4_grouped_gemm_fc1_swiglu(a_codes, a_sf, a_g, offsets, E, M_cap, d, d_ff, w1_codes, w1_sf, w1_g,
                                  h_codes, h_sf, h_g, dbg_u_f32, dbg_h, ws, status=None, stream=None):
    _check("nvfp4_grouped_gemm_fc1_swiglu", lib().nvfp4_grouped_gemm_fc1_swiglu(
        _p(a_codes), _p(a_sf), _p(a_g), _p(offsets), E, M_cap, d, d_ff, _p(w1_codes), _p(w1_sf), _p(w1_g),
        _p(h_codes), _p(h_sf), _p(h_g), _p(dbg_u_f32), _p(dbg_h), _p(ws),
        ws.numel() * ws.element_size(), _p(status), _s(stream)))


def nvfp4_grouped_gemm_fc2_unpermute(h_codes, h_sf, h_g, offsets, E, M_cap, d_ff, d, w2_codes, w2_sf, w2_g,
                                     row_to_token, token_slot_row, topk_w, T, k, slots, out, dbg_y_f32,
                                     status=None, stream=None):
    """slots: the z rows, bf16 [M_cap][d] (the kernel stores whole 128-row
    tiles there)."""
    if T > 0 and slots.numel() * slots.element_size() < M_cap * d * 2:
        raise ValueError("slots must hold M_cap x d bf16 values")
    _check("nvfp4_grouped_gemm_fc2_unpermute", lib().nvfp4_grouped_gemm_fc2_unpermute(
        _p(h_codes), _p(h_sf), _p(h_g), _p(offsets), E, M_cap, d_ff, d, _p(w2_codes), _p(w2_sf), _p(w2_g),
        _p(row_to_token), _p(token_slot_row), _p(topk_w), T, k, _p(slots), _p(out), _p(dbg_y_f32),
        _p(status), _s(stream)))


def moe_expert_forward(x, logits, T, E, k, d, d_ff, w1_codes, w1_sf, w1_g, w2_codes, w2_sf, w2_g, out, ws,
                       status=None, stream=None):
    _check("moe_expert_forward", lib().moe_expert_forward(
        _p(x), _p(logits), T, E, k, d, d_ff, _p(w1_codes), _p(w1_sf), _p(w1_g), _p(w2_codes), _p(w2_sf),
        _p(w2_g), _p(out), _p(ws), 0 if ws is None else ws.numel() * ws.element_size(), _p(status),
        _s(stream)))


def moe_expert_forward_timed(x, logits, T, E, k, d, d_ff, w1_codes, w1_sf, w1_g, w2_codes, w2_sf, w2_g, out, ws,
                             status=None, stream=None, events=None):
    """moe_expert_forward recording the eight torch.cuda.Event objects in
    `events` (timing enabled) around its seven launches on the stream."""
    import torch
    if events is None or len(events) != 8:
        raise ValueError("events: eight torch.cuda.Event objects")
    s = torch.cuda.current_stream() if stream is None else stream
    for e in events:  # the handle exists once the event has been recorded
        if e.cuda_event == 0:
            e.record(s)
    arr = (ctypes.c_void_p * 8)(*[e.cuda_event for e in events])
    _check("moe_expert_forward_timed", lib().moe_expert_forward_timed(
        _p(x), _p(logits), T, E, k, d, d_ff, _p(w1_codes), _p(w1_sf), _p(w1_g), _p(w2_codes), _p(w2_sf),
        _p(w2_g), _p(out), _p(ws), 0 if ws is None else ws.numel() * ws.element_size(), _p(status),
        _s(stream), ctypes.cast(arr, P)))


def moe_expert_forward_gather(x, logits, T, E, k, d, d_ff, w1_codes, w1_sf, w1_g, w2_codes, w2_sf, w2_g, out, ws,
                              status=None, stream=None):
    """moe_expert_forward with gather-on-load FC1 (codes quantised once per
    token, fetched by row_to_token with TMA tile::gather4)."""
    _check("moe_expert_forward_gather", lib().moe_expert_forward_gather(
        _p(x), _p(logits), T, E, k, d, d_ff, _p(w1_codes), _p(w1_sf), _p(w1_g), _p(w2_codes), _p(w2_sf),
        _p(w2_g), _p(out), _p(ws), 0 if ws is None else ws.numel() * ws.element_size(), _p(status),
        _s(stream)))


def moe_expert_forward_train(x, logits, T, E, k, d, d_ff, w1_codes, w1_sf, w1_g, w2_codes, w2_sf, w2_g, out, ws,
                             save_u, save_h, status=None, stream=None):
    _check("moe_expert_forward_train", lib().moe_expert_forward_train(
        _p(x), _p(logits), T, E, k, d, d_ff, _p(w1_codes), _p(w1_sf), _p(w1_g), _p(w2_codes), _p(w2_sf),
        _p(w2_g), _p(out), _p(ws), 0 if ws is None else ws.numel() * ws.element_size(), _p(save_u), _p(save_h),
        _p(status), _s(stream)))


def moe_expert_backward(dY, x, T, E, k, d, d_ff, W1, W2, w2_codes, w2_sf, w2_g, topk_ids, topk_w, offsets,
                        row_to_token, token_slot_row, u, h, h_codes, h_sf, h_g, dx, dW1, dW2, dlogits, dw, ws,
                        status=None, stream=None):
    _check("moe_expert_backward", lib().moe_expert_backward(
        _p(dY), _p(x), T, E, k, d, d_ff, _p(W1), _p(W2), _p(w2_codes), _p(w2_sf), _p(w2_g), _p(topk_ids),
        _p(topk_w), _p(offsets), _p(row_to_token), _p(token_slot_row), _p(u), _p(h), _p(h_codes), _p(h_sf),
        _p(h_g), _p(dx), _p(dW1), _p(dW2), _p(dlogits), _p(dw), _p(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _p(status), _s(stream)))


def backward_workspace_bytes(T, E, k, d, d_ff):
    return int(lib().moe_expert_backward_workspace_bytes(T, E, k, d, d_ff))


class Pipeline:
    """moe_pipeline_*: the forward on host-resident batches, with the copies
    of neighbouring steps overlapping the forward (three streams, `depth`
    slots).  Host tensors should be pinned."""

    def __init__(self, T, E, k, d, d_ff, depth=2, device="cuda"):
        import torch
        n = int(lib().moe_pipeline_device_bytes(T, E, k, d, d_ff, depth))
        if n == 0:
            raise MoeError("moe_pipeline_device_bytes", MOE_ERR_SHAPE)
        self.buf = torch.empty(n + 1024, dtype=torch.uint8, device=device)
        off = (-self.buf.data_ptr()) % 1024
        self._h = ctypes.c_void_p()
        _check("moe_pipeline_create", lib().moe_pipeline_create(
            T, E, k, d, d_ff, depth, ctypes.c_void_p(self.buf.data_ptr() + off), n, ctypes.byref(self._h)))

    def submit(self, x_host, logits_host, out_host, w1q, w2q, status=None):
        _check("moe_pipeline_submit", lib().moe_pipeline_submit(
            self._h, _p(x_host), _p(logits_host), _p(out_host), _p(w1q["codes"]), _p(w1q["sf"]), _p(w1q["g"]),
            _p(w2q["codes"]), _p(w2q["sf"]), _p(w2q["g"]), _p(status)))

    def synchronize(self):
        _check("moe_pipeline_synchronize", lib().moe_pipeline_synchronize(self._h))

    def close(self):
        if self._h:
            rc = lib().moe_pipeline_destroy(self._h)
            self._h = ctypes.c_void_p()
            _check("moe_pipeline_destroy", rc)


# --------------------------------------------------------------------------
# device-memory helpers (torch allocations of the buffers the calls expect)
# --------------------------------------------------------------------------
def empty_quantized(rows, K, device="cuda"):
    import torch
    return dict(codes=torch.empty((rows, K // 2), dtype=torch.uint8, device=device),
                sf=torch.empty(max(sf_bytes(rows, K), 16), dtype=torch.uint8, device=device),
                g=torch.empty(rows, dtype=torch.float32, device=device))


def quantize_weights(W):
    """Quantise expert weights W [E][N][K] (bf16) on the GPU; returns a dict
    with codes [E][N][K/2], sf (flat) and g [E][N]."""
    E, N, K = W.shape
    q = empty_quantized(E * N, K, W.device)
    moe_nvfp4_quantize_weights(W, q["codes"], q["sf"], q["g"])
    q["codes"] = q["codes"].view(E, N, K // 2)
    q["g"] = q["g"].view(E, N)
    return q


def quantize_weights_per_expert(W):
    """quantize_weights with one outer scale per expert tensor; the dict also
    holds amax_e [E] = max |W_e|."""
    import torch
    E, N, K = W.shape
    q = empty_quantized(E * N, K, W.device)
    q["amax_e"] = torch.empty(E, dtype=torch.float32, device=W.device)
    moe_nvfp4_quantize_weights_per_expert(W, q["codes"], q["sf"], q["g"], q["amax_e"])
    q["codes"] = q["codes"].view(E, N, K // 2)
    q["g"] = q["g"].view(E, N)
    return q


def forward_workspace(T, E, k, d, d_ff, device="cuda"):
    import torch
    n = forward_workspace_bytes(T, E, k, d, d_ff)
    if n == 0:
        raise MoeError("moe_expert_forward_workspace_bytes", MOE_ERR_SHAPE)
    return torch.empty(n, dtype=torch.uint8, device=device)


def forward_views(ws, T, E, k, d, d_ff):
    """Typed views of the intermediates that moe_expert_forward leaves in ws."""
    import torch
    lay = forward_workspace_layout(T, E, k, d, d_ff)
    mc = m_cap(T, E, k)

    def v(name, dtype, shape, nbytes=None):
        o = lay[name]
        esz = torch.empty((), dtype=dtype).element_size()
        n = 1
        for s in shape:
            n *= s
        return ws[o:o + n * esz].view(dtype).view(*shape)

    return dict(
        topk_ids=v("topk_ids", torch.int32, (T, k)), topk_w=v("topk_w", torch.float32, (T, k)),
        token_slot_row=v("token_slot_row", torch.int32, (T, k)), counts=v("counts", torch.int32, (E,)),
        offsets=v("offsets", torch.int32, (E + 1,)), row_to_token=v("row_to_token", torch.int32, (mc,)),
        amax_tok=v("amax_tok", torch.float32, (T,)), x_codes=v("x_codes", torch.uint8, (mc, d // 2)),
        x_sf=v("x_sf", torch.uint8, (sf_bytes(mc, d),)), x_g=v("x_g", torch.float32, (mc,)),
        h_codes=v("h_codes", torch.uint8, (mc, d_ff // 2)), h_sf=v("h_sf", torch.uint8, (sf_bytes(mc, d_ff),)),
        h_g=v("h_g", torch.float32, (mc,)), slots=v("slots", torch.int16, (mc, d)), m_cap=mc)
