"""Exhaustive parity of the GPU codecs with the oracle: every non-negative
finite float is encoded on the GPU; monotonicity plus equal first inputs of
every code make the two encoders identical on all finite inputs."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_codecs_exhaustive(orc):
    from gpu_util import build_test_so
    L = ctypes.CDLL(build_test_so("codec_sweep"))
    f4 = (ctypes.c_uint * 128)()
    f2 = (ctypes.c_uint * 8)()
    v4, v2, vs = ctypes.c_ulonglong(), ctypes.c_ulonglong(), ctypes.c_ulonglong()
    vals = (ctypes.c_float * 128)()
    assert L.run_codec_sweeps(f4, ctypes.byref(v4), f2, ctypes.byref(v2), ctypes.byref(vs), vals) == 0
    assert v4.value == 0 and v2.value == 0 and vs.value == 0
    for c in range(1, 0x7F):
        assert f4[c] == orc.lib().orc_e4m3_first_input_of_code(c), hex(c)
    for c in range(1, 8):
        assert f2[c] == orc.lib().orc_e2m1_first_input_of_code(c), c
    for c in range(0x7F):
        assert vals[c] == orc.e4m3_value(c)


def test_hardware_e2m1_conversion_exhaustive(orc):
    """The quantisers encode with the hardware E2M1 conversion; it equals the
    reference encoder (itself equal to the oracle above) on every finite
    float of either sign."""
    from gpu_util import build_test_so
    L = ctypes.CDLL(build_test_so("codec_sweep"))
    v = ctypes.c_ulonglong()
    assert L.run_cvt_sweep(ctypes.byref(v)) == 0
    assert v.value == 0


def test_quantiser_fast_paths_exhaustive():
    """The quantisers' fast paths equal their exact definitions: the
    hardware E4M3 conversion and decode (every non-negative finite float,
    every code); the bracketed block scale E4M3(RN(a / den)) (every finite
    BF16 amax with 65536 divisors across the float range); and the E2M1
    encoder, Q(RN(v / S)) for every finite BF16 value up to 16 S with 65536
    scales across the float range, each under three row scales (Markstein's
    division after the row's power-of-two factor)."""
    from gpu_util import build_test_so
    L = ctypes.CDLL(build_test_so("codec_sweep"))
    v1, v2, v3 = ctypes.c_ulonglong(), ctypes.c_ulonglong(), ctypes.c_ulonglong()
    assert L.run_fast_path_sweeps(ctypes.byref(v1), ctypes.byref(v2), ctypes.byref(v3)) == 0
    print("e4m3 hw mismatches %d, block-scale mismatches %d, e2m1 encoder mismatches %d"
          % (v1.value, v2.value, v3.value))
    assert v1.value == 0 and v2.value == 0 and v3.value == 0


def test_markstein_division_codes_exhaustive():
    """The quantisers' E2M1 codes come from Markstein's correctly rounded
    division (RN(1/S) once per block, then two FMA corrections of v RN(1/S))
    with no fallback: inside its domain (row factor 1) its codes equal
    Q(RN(v / S)) from the IEEE division for
    every finite BF16 v (either sign) within its domain |v| <= 16 S, over
    65536 scales across [2^-96, 2^120], all-ones significands at every
    exponent among them."""
    from gpu_util import build_test_so
    L = ctypes.CDLL(build_test_so("codec_sweep"))
    viol, checked = ctypes.c_ulonglong(), ctypes.c_ulonglong()
    assert L.run_div_sweep(ctypes.byref(viol), ctypes.byref(checked)) == 0
    print("markstein division: %d (v, S) pairs, %d mismatching 8-value groups" % (checked.value, viol.value))
    assert checked.value > 2 ** 31  # the domain holds most (v, S) pairs
    assert viol.value == 0

