"""MOE-NVFP4-SPEC-1 oracle: numpy front end of the plain C++ CPU restatement.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` (``cpu_baseline`` and ``--impl reference``) may import
this package.  The CUDA library and its Python binding never import it, and it
imports nothing from them.

Each function composes the C steps of ``oracle.cpp`` in the order the pages
give them (see the citation tags in ``oracle.h``):

  route -> permute -> amax -> quantise (per token, k copies) -> grouped FC1
  -> BF16 cast + SwiGLU -> requantise h -> grouped FC2 -> router-weighted
  BF16 scatter -> ascending-expert-id reduce.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I32 = ctypes.c_int
I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (IEEE binary32, no contraction, no FTZ)."""
    src = os.path.join(_HERE, "oracle.cpp")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(src),
                                                   os.path.getmtime(os.path.join(_HERE, "oracle.h")))):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-fPIC", "-shared", src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            sig = {
                "orc_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "orc_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
                "orc_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
                "orc_e2m1_value": (ctypes.c_float, [ctypes.c_uint8]),
                "orc_e2m1_encode": (ctypes.c_uint8, [ctypes.c_float]),
                "orc_e4m3_value": (ctypes.c_float, [ctypes.c_uint8]),
                "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
                "orc_sf_offset": (I64, [I64, I64, I64]),
                "orc_sf_bytes": (I64, [I64, I64]),
                "orc_m_cap": (I64, [I64, I64, I64]),
                "orc_unswizzle_sf": (None, [P, I64, I32, P]),
                "orc_quantize_row": (None, [P, I32, ctypes.c_float, P, P, P]),
                "orc_amax_rows_bf16": (None, [P, I64, I32, P]),
                "orc_quantize_rows_bf16": (None, [P, I64, I32, P, P, I64, P, P, P]),
                "orc_dequantize_rows": (None, [P, P, P, I64, I32, P]),
                "orc_route": (I32, [P, I64, I32, I32, P, P]),
                "orc_permute": (I32, [P, I64, I32, I32, I64, P, P, P, P]),
                "orc_grouped_gemm": (None, [P, P, P, P, I32, I64, I32, I32, P, P, P, P]),
                "orc_swiglu": (None, [P, I64, I32, P, P]),
                "orc_combine": (None, [P, P, P, P, I64, I32, I64, I32, P]),
                "orc_reduce": (None, [P, I64, I32, I32, P]),
                "orc_e4m3_first_input_of_code": (I64, [ctypes.c_uint8]),
                "orc_e2m1_first_input_of_code": (I64, [ctypes.c_uint8]),
                "orc_num_threads": (I32, []),
                "orc_set_num_threads": (None, [I32]),
                "orc_rht16_rows": (None, [P, I64, I32, P, P]),
                "orc_quantize_tensor": (None, [P, I64, I32, P, P, P]),
                "orc_quantize_weights_per_expert": (None, [P, I32, I32, I32, P, P, P]),
                "orc_bwd_router": (None, [P, P, P, P, P, I64, I32, I32, I32, P, P]),
                "orc_bwd_dy2": (None, [P, P, P, I64, I32, I32, I64, P]),
                "orc_bwd_expert": (None, [P, P, P, P, I64, I32, I32, P, P, P, P, P, P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# scalar and vector codecs
# --------------------------------------------------------------------------
def bf16_bits_to_f32(b):
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x):
    x = _c(x, np.float32)
    f = lib().orc_f32_to_bf16
    out = np.empty(x.shape, np.uint16)
    flat, oflat = x.reshape(-1), out.reshape(-1)
    for i in range(flat.size):
        oflat[i] = f(float(flat[i]))
    return out


def e2m1_value(code):
    return lib().orc_e2m1_value(int(code))


def e2m1_encode(q):
    return lib().orc_e2m1_encode(float(np.float32(q)))


def e4m3_value(code):
    return lib().orc_e4m3_value(int(code))


def e4m3_encode(t):
    return lib().orc_e4m3_encode(float(np.float32(t)))


def sf_bytes(rows, K):
    return int(lib().orc_sf_bytes(rows, K))


def m_cap(T, E, k):
    return int(lib().orc_m_cap(T, E, k))


def sf_offset(row, col, K):
    return int(lib().orc_sf_offset(row, col, K))


def unswizzle_sf(sf_swz, rows, K):
    """Logical [rows][K/16] view of a swizzled scale buffer (oracle layout)."""
    sf = _c(sf_swz, np.uint8)
    out = np.zeros((rows, K // 16), np.uint8)
    lib().orc_unswizzle_sf(_p(sf), rows, K, _p(out))
    return out


# --------------------------------------------------------------------------
# quantisation
# --------------------------------------------------------------------------
def quantize_row(v, amax=None):
    v = _c(v, np.float32)
    K = v.size
    a = float(np.max(np.abs(v))) if amax is None else float(amax)
    codes = np.zeros(K // 2, np.uint8)
    sf = np.zeros(K // 16, np.uint8)
    g = np.zeros(1, np.float32)
    lib().orc_quantize_row(_p(v), K, a, _p(codes), _p(sf), _p(g))
    return codes, sf, float(g[0])


def amax_rows(x_bf16):
    x = _c(x_bf16, np.uint16)
    rows, K = x.shape
    out = np.zeros(rows, np.float32)
    lib().orc_amax_rows_bf16(_p(x), rows, K, _p(out))
    return out


def quantize_rows(src_bf16, row_map=None, amax=None, dst_rows=None):
    """Returns (codes [dst][K/2] u8, sf_swz [sf_bytes] u8, g [dst] f32)."""
    src = _c(src_bf16, np.uint16)
    src_rows, K = src.shape
    if dst_rows is None:
        dst_rows = src_rows if row_map is None else len(row_map)
    rm = None if row_map is None else _c(row_map, np.int32)
    am = None if amax is None else _c(amax, np.float32)
    codes = np.zeros((dst_rows, K // 2), np.uint8)
    sf = np.zeros(max(sf_bytes(dst_rows, K), 1), np.uint8)
    g = np.zeros(dst_rows, np.float32)
    lib().orc_quantize_rows_bf16(_p(src), src_rows, K, _p(rm), _p(am), dst_rows,
                                 _p(codes), _p(sf), _p(g))
    return codes, sf, g


def dequantize_rows(codes, sf_swz, g, K):
    codes = _c(codes, np.uint8)
    rows = codes.shape[0]
    out = np.zeros((rows, K), np.float64)
    lib().orc_dequantize_rows(_p(codes), _p(_c(sf_swz, np.uint8)),
                              _p(_c(g, np.float32)), rows, K, _p(out))
    return out


# --------------------------------------------------------------------------
# routing, permutation, GEMM, epilogues
# --------------------------------------------------------------------------
def route(logits, k):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    rc = lib().orc_route(_p(logits), T, E, k, _p(ids), _p(w))
    if rc != 0:
        raise ValueError("non-finite router logit")
    return ids, w


def permute(ids, E):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    mc = m_cap(T, E, k)
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    r2t = np.full(max(mc, 1), -1, np.int32)[:mc]
    tsr = np.zeros((T, k), np.int32)
    m_pad = lib().orc_permute(_p(ids), T, E, k, mc, _p(counts), _p(offsets),
                              _p(r2t), _p(tsr))
    if m_pad < 0:
        raise ValueError("bad expert id")
    return dict(counts=counts, offsets=offsets, row_to_token=r2t,
                token_slot_row=tsr, m_pad=int(m_pad), m_cap=mc)


def grouped_gemm(a_codes, a_sf, a_g, offsets, w_codes, w_sf, w_g, K, N):
    a_codes = _c(a_codes, np.uint8)
    M = a_codes.shape[0]
    offsets = _c(offsets, np.int32)
    E = offsets.size - 1
    y = np.zeros((M, N), np.float32)
    lib().orc_grouped_gemm(_p(a_codes), _p(_c(a_sf, np.uint8)), _p(_c(a_g, np.float32)),
                           _p(offsets), E, M, K, N, _p(_c(w_codes, np.uint8)),
                           _p(_c(w_sf, np.uint8)), _p(_c(w_g, np.float32)), _p(y))
    return y


def swiglu(y, F):
    y = _c(y, np.float32)
    M = y.shape[0]
    u = np.zeros((M, 2 * F), np.uint16)
    h = np.zeros((M, F), np.uint16)
    lib().orc_swiglu(_p(y), M, F, _p(u), _p(h))
    return u, h


def combine(y2, perm, topk_w, T, k, d):
    y2 = _c(y2, np.float32)
    slots = np.zeros((T, k, d), np.uint16)
    lib().orc_combine(_p(y2), _p(perm["row_to_token"]), _p(perm["token_slot_row"]),
                      _p(_c(topk_w, np.float32)), T, k, y2.shape[0], d, _p(slots))
    return slots


def reduce(slots):
    slots = _c(slots, np.uint16)
    T, k, d = slots.shape
    out = np.zeros((T, d), np.uint16)
    lib().orc_reduce(_p(slots), T, k, d, _p(out))
    return out


def quantize_weights(W_bf16):
    """Per-output-row quantisation of expert weights W [E][N][K] (BF16 bits)."""
    W = _c(W_bf16, np.uint16)
    E, N, K = W.shape
    codes, sf, g = quantize_rows(W.reshape(E * N, K))
    return codes.reshape(E, N, K // 2), sf, g.reshape(E, N)


def moe_forward(x_bf16, logits, w1q, w2q, k, d_ff, ext_ids=None, ext_w=None):
    """Full expert forward; returns every intermediate of the specification.

    w1q / w2q are (codes, sf_swz, g) from quantize_weights of W1 [E][2 d_ff][d]
    and W2 [E][d][d_ff].  ext_ids / ext_w replace the router (routing replay).
    """
    x = _c(x_bf16, np.uint16)
    T, d = x.shape
    E = w1q[2].shape[0]
    if ext_ids is None:
        ids, w = route(logits, k)
    else:
        ids, w = _c(ext_ids, np.int32), _c(ext_w, np.float32)
    perm = permute(ids, E)
    amax_tok = amax_rows(x)
    mc = perm["m_cap"]
    x_codes, x_sf, x_g = quantize_rows(x, perm["row_to_token"], amax_tok, mc)
    y1 = grouped_gemm(x_codes, x_sf, x_g, perm["offsets"], w1q[0], w1q[1], w1q[2],
                      d, 2 * d_ff)
    u, h = swiglu(y1, d_ff)
    h_codes, h_sf, h_g = quantize_rows(h)
    y2 = grouped_gemm(h_codes, h_sf, h_g, perm["offsets"], w2q[0], w2q[1], w2q[2],
                      d_ff, d)
    slots = combine(y2, perm, w, T, k, d)
    out = reduce(slots)
    amax_row = np.where(perm["row_to_token"] >= 0,
                        amax_tok[np.maximum(perm["row_to_token"], 0)], 0).astype(np.float32)
    return dict(ids=ids, w=w, perm=perm, amax_tok=amax_tok, amax_row=amax_row,
                x_codes=x_codes, x_sf=x_sf, x_g=x_g, y1=y1, u=u, h=h,
                h_codes=h_codes, h_sf=h_sf, h_g=h_g, y2=y2, slots=slots, out=out)


class TokenOracle:
    """Output of single tokens of a large layer, computed one by one.

    Used where the full layer is too large for the oracle: the token is routed
    alone, quantised alone (its codes do not depend on other tokens, the
    context-swap property of per-token scaling), and run through its k experts
    with weights the oracle quantises itself, expert by expert, on demand.
    """

    def __init__(self, W1_bf16, W2_bf16, k):
        self.W1, self.W2, self.k = W1_bf16, W2_bf16, k
        self.E, self.N1, self.d = W1_bf16.shape
        self.d_ff = self.N1 // 2
        self._cache = {}

    def _wq(self, e):
        if e not in self._cache:
            self._cache[e] = (quantize_weights(self.W1[e:e + 1]),
                              quantize_weights(self.W2[e:e + 1]))
        return self._cache[e]

    def token(self, x_row_bf16, logits_row):
        k, d, F = self.k, self.d, self.d_ff
        ids, w = route(np.asarray(logits_row, np.float32)[None, :], k)
        xr = _c(x_row_bf16, np.uint16)[None, :]
        xc, xs, xg = quantize_rows(xr)
        res = dict(ids=ids[0], w=w[0], y1=[], h=[], y2=[], x_codes=xc[0], x_g=xg[0])
        for j in range(k):
            e = int(ids[0, j])
            (w1c, w1s, w1g), (w2c, w2s, w2g) = self._wq(e)
            off = np.array([0, 1], np.int32)
            y1 = grouped_gemm(xc, xs, xg, off, w1c, w1s, w1g, d, 2 * F)
            _, h = swiglu(y1, F)
            hc, hs, hg = quantize_rows(h)
            y2 = grouped_gemm(hc, hs, hg, off, w2c, w2s, w2g, F, d)
            res["y1"].append(y1[0])
            res["h"].append(h[0])
            res["y2"].append(y2[0])
        y2 = np.stack(res["y2"])
        one = dict(row_to_token=np.zeros(k, np.int32),
                   token_slot_row=np.arange(k, dtype=np.int32)[None, :])
        slots = combine(y2, one, w, 1, k, d)
        res["slots"] = slots[0]
        res["out"] = reduce(slots)[0]
        return res


def num_threads():
    return int(lib().orc_num_threads())


def set_num_threads(n):
    """Threads of the oracle's parallel loops from now on; results do not
    depend on it."""
    lib().orc_set_num_threads(int(n))


# --------------------------------------------------------------------------
# contrast recipes (not the hot path's recipe)
# --------------------------------------------------------------------------
def rht16_rows(x_f32, signs16):
    """Blockwise 16-point random Hadamard transform of FP32 rows."""
    x = _c(x_f32, np.float32)
    rows, K = x.shape
    y = np.zeros_like(x)
    lib().orc_rht16_rows(_p(x), rows, K, _p(_c(signs16, np.int8)), _p(y))
    return y


def quantize_tensor(x_f32):
    """Per-tensor NVFP4: (codes, sf_swz, g [rows]) with one shared g."""
    x = _c(x_f32, np.float32)
    rows, K = x.shape
    codes = np.zeros((rows, K // 2), np.uint8)
    sf = np.zeros(max(sf_bytes(rows, K), 1), np.uint8)
    g = np.zeros(rows, np.float32)
    lib().orc_quantize_tensor(_p(x), rows, K, _p(codes), _p(sf), _p(g))
    return codes, sf, g


def quantize_per_tensor_rht(x_bf16, signs16):
    """The RHT-enabled per-tensor contrast reference: BF16 rows -> FP32 ->
    blockwise RHT -> per-tensor NVFP4."""
    x = bf16_bits_to_f32(_c(x_bf16, np.uint16))
    return quantize_tensor(rht16_rows(x, signs16))


def quantize_weights_per_expert(W_bf16):
    """Weights [E][N][K] (BF16 bits) with one outer scale per expert tensor:
    (codes [E][N][K/2], sf_swz, g [E][N] with g[e][:] = g_e)."""
    W = _c(W_bf16, np.uint16)
    E, N, K = W.shape
    codes = np.zeros((E, N, K // 2), np.uint8)
    sf = np.zeros(max(sf_bytes(E * N, K), 1), np.uint8)
    g = np.zeros((E, N), np.float32)
    lib().orc_quantize_weights_per_expert(_p(W), E, N, K, _p(codes), _p(sf), _p(g))
    return codes, sf, g


# --------------------------------------------------------------------------
# backward: straight-through estimator, BF16 GEMM operands (orc_bwd_* in
# oracle.h state the formulas and the passages they follow)
# --------------------------------------------------------------------------
def bwd_router(dY_bf16, y2, w, ids, token_slot_row, E):
    dY = _c(dY_bf16, np.uint16)
    T, d = dY.shape
    k = ids.shape[1]
    dw = np.zeros((T, k), np.float32)
    dl = np.zeros((T, E), np.float32)
    lib().orc_bwd_router(_p(dY), _p(_c(y2, np.float32)), _p(_c(w, np.float32)), _p(_c(ids, np.int32)),
                         _p(_c(token_slot_row, np.int32)), T, k, d, E, _p(dw), _p(dl))
    return dw, dl


def bwd_dy2(dY_bf16, w, token_slot_row, M):
    dY = _c(dY_bf16, np.uint16)
    T, d = dY.shape
    k = w.shape[1]
    out = np.zeros((M, d), np.uint16)
    lib().orc_bwd_dy2(_p(dY), _p(_c(w, np.float32)), _p(_c(token_slot_row, np.int32)), T, k, d, M, _p(out))
    return out


def bwd_expert(dy2_rows, u_rows, h_rows, x_rows, W1e, W2e):
    """One expert over the given rows: (du BF16 [n][2F], dxr FP64 [n][d],
    dW1 FP32 [2F][d], dW2 FP32 [d][F])."""
    dy2 = _c(dy2_rows, np.uint16)
    n, d = dy2.shape
    F = W2e.shape[1]
    du = np.zeros((n, 2 * F), np.uint16)
    dxr = np.zeros((n, d), np.float64)
    dW1 = np.zeros((2 * F, d), np.float32)
    dW2 = np.zeros((d, F), np.float32)
    lib().orc_bwd_expert(_p(dy2), _p(_c(u_rows, np.uint16)), _p(_c(h_rows, np.uint16)), _p(_c(x_rows, np.uint16)),
                         n, d, F, _p(_c(W1e, np.uint16)), _p(_c(W2e, np.uint16)), _p(du), _p(dxr), _p(dW1), _p(dW2))
    return du, dxr, dW1, dW2


def gather_x_rows(x_bf16, row_to_token):
    """BF16 input row of each permuted row's token, zero on pad rows (a
    gather, no arithmetic)."""
    x = _c(x_bf16, np.uint16)
    r2t = np.asarray(row_to_token)
    out = np.zeros((r2t.shape[0], x.shape[1]), np.uint16)
    real = r2t >= 0
    out[real] = x[r2t[real]]
    return out


def moe_backward(dY_bf16, x_bf16, W1_bf16, W2_bf16, fwd):
    """Straight-through backward of moe_forward's result `fwd` (its ids, w,
    permutation, u, h and y2 are the saved values).  Returns dx FP32 [T][d]
    (sum over the token's slots in FP64, rounded once), dW1 FP32 [E][2F][d],
    dW2 FP32 [E][d][F], dw FP32 [T][k], dlogits FP32 [T][E], and the BF16
    GEMM operands dy2 [M][d] and du [M][2F] (M = padded rows)."""
    W1, W2 = _c(W1_bf16, np.uint16), _c(W2_bf16, np.uint16)
    E, F2, d = W1.shape
    F = F2 // 2
    perm = fwd["perm"]
    M = perm["m_pad"]
    offs = perm["offsets"]
    T = x_bf16.shape[0]
    dw, dl = bwd_router(dY_bf16, fwd["y2"], fwd["w"], fwd["ids"], perm["token_slot_row"], E)
    dy2 = bwd_dy2(dY_bf16, fwd["w"], perm["token_slot_row"], M)
    xr = gather_x_rows(x_bf16, perm["row_to_token"][:M])
    du = np.zeros((M, F2), np.uint16)
    dxr = np.zeros((M, d), np.float64)
    dW1 = np.zeros((E, F2, d), np.float32)
    dW2 = np.zeros((E, d, F), np.float32)
    u, h = np.asarray(fwd["u"]), np.asarray(fwd["h"])
    for e in range(E):
        a, b = int(offs[e]), int(offs[e + 1])
        if a == b:
            continue
        du[a:b], dxr[a:b], dW1[e], dW2[e] = bwd_expert(dy2[a:b], u[a:b], h[a:b], xr[a:b], W1[e], W2[e])
    tsr = perm["token_slot_row"]
    dx = dxr[tsr].sum(axis=1).astype(np.float32) if T > 0 else np.zeros((0, d), np.float32)
    return dict(dx=dx, dW1=dW1, dW2=dW2, dw=dw, dlogits=dl, dy2=dy2, du=du, dxr=dxr)
