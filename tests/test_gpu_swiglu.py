"""The FC1 epilogue's SwiGLU, h = BF16(silu(g) * up) rounded once, against
the oracle and exhaustively.

The epilogue decides most elements with a bracket around a fast FP32 value
whose error bound rests on the hardware ex2/rcp approximations; the rest go
to a double-float evaluation and, within 2^-40 of a rounding midpoint, to
FP64 (swiglu.cuh).  Checked here:
  - the hardware approximation errors, measured over every input the
    bracket can see, fit inside the bracket's half-width;
  - over all 2^32 pairs of finite BF16 values, the epilogue's function and
    the double-float tier alone both equal the FP64 tier bit for bit;
  - every finite BF16 gate value with 64 seeded up values equals the CPU
    oracle's SwiGLU bit for bit.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _lib():
    from gpu_util import build_test_so
    L = ctypes.CDLL(build_test_so("swiglu_sweep"))
    L.swiglu_eps.restype = ctypes.c_float
    L.swiglu_c1.restype = ctypes.c_float
    L.swiglu_c2ln2.restype = ctypes.c_float
    return L


def test_bracket_covers_hardware_error():
    L = _lib()
    e_ex2, e_rcp = ctypes.c_float(), ctypes.c_float()
    assert L.run_hw_bounds(ctypes.byref(e_ex2), ctypes.byref(e_rcp)) == 0
    # relative error bound of the fast value p: ex2 of the exact argument
    # g * C1; the first-order factor 1 + g C2 ln 2 drops (g C2 ln 2)^2 / 2
    # for |g| up to 128 / |C1| (beyond, E overflows and p is flagged) and
    # rounds once (fma); the reciprocal; the roundings of 1 + E, g * r and p;
    # plus 2^-24 for the rounding of the bracket products
    c1, c2 = abs(L.swiglu_c1()), abs(L.swiglu_c2ln2())
    assert c1 * 2 ** 15 == int(c1 * 2 ** 15) and int(c1 * 2 ** 15) < 2 ** 16  # 16 significant bits
    assert abs(c1 + c2 / np.log(2) - 1 / np.log(2)) < 1e-12  # C1 + C2 = log2 e
    dmax = 128.0 / c1 * c2
    bound = e_ex2.value + dmax ** 2 / 2 + 2.0 ** -24 + e_rcp.value + 3 * 2.0 ** -24 + 2.0 ** -24
    print("ex2.approx.ftz max rel %.3e, rcp.approx.ftz max rel %.3e, needed eps %.3e, eps %.3e"
          % (e_ex2.value, e_rcp.value, bound, L.swiglu_eps()))
    assert 0 < e_ex2.value < 1e-5 and 0 < e_rcp.value < 1e-5
    assert bound <= L.swiglu_eps()


def test_swiglu_all_bf16_pairs():
    L = _lib()
    bad, open_n, tested, bad2 = (ctypes.c_ulonglong() for _ in range(4))
    assert L.run_sweep_all(ctypes.byref(bad), ctypes.byref(open_n), ctypes.byref(tested), ctypes.byref(bad2)) == 0
    n_finite = 65536 - 2 * 128
    assert tested.value == n_finite * n_finite
    print("all pairs: %d mismatches, tier 2 alone %d mismatches; bracket open on %.3e of the pairs"
          % (bad.value, bad2.value, open_n.value / tested.value))
    assert bad.value == 0 and bad2.value == 0
    # over all pairs the bracket leaves well under 1% open: besides
    # straddles of a midpoint, for large g the product g * up of two 8-bit
    # significands is often itself a BF16 midpoint, which p * (1 -+ eps)
    # always straddles
    assert open_n.value / tested.value < 1e-2


def test_swiglu_against_oracle(orc):
    L = _lib()
    gs = np.arange(65536, dtype=np.uint32)
    gs = gs[(gs & 0x7F80) != 0x7F80].astype(np.uint16)  # finite BF16 values
    rng = np.random.default_rng(0)
    ups = rng.integers(0, 65536, 64, dtype=np.uint32)
    ups = np.where((ups & 0x7F80) == 0x7F80, ups & 0x807F, ups).astype(np.uint16)
    g = np.repeat(gs, len(ups))
    up = np.tile(ups, len(gs))
    n = (len(g) + 15) // 16 * 16
    g = np.concatenate([g, np.zeros(n - len(g), np.uint16)])
    up = np.concatenate([up, np.zeros(n - len(up), np.uint16)])
    h = np.zeros(n, np.uint16)
    P = ctypes.POINTER(ctypes.c_uint16)
    assert L.run_eval_pairs(g.ctypes.data_as(P), up.ctypes.data_as(P), h.ctypes.data_as(P), n) == 0
    # the oracle's SwiGLU takes FC1 outputs [rows][2F] (gate then up); BF16
    # values pass its cast unchanged
    f32 = lambda b: (b.astype(np.uint32) << 16).view(np.float32)
    y = np.stack([f32(g), f32(up)], axis=1).astype(np.float32)
    _, h_ref = orc.swiglu(y, 1)
    assert np.array_equal(h, h_ref.reshape(-1))
