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
    BF16 amax with 65536 divisors across the float range); the bracketed
    E2M1 codes Q(RN(v / S)) (every finite BF16 value with 65536 scales); and
    the hardware reciprocal the E2M1 bracket rests on stays within 2^-23
    relative over the bracket's domain."""
    from gpu_util import build_test_so
    L = ctypes.CDLL(build_test_so("codec_sweep"))
    v1, v2, v3 = ctypes.c_ulonglong(), ctypes.c_ulonglong(), ctypes.c_ulonglong()
    e = ctypes.c_float()
    assert L.run_fast_path_sweeps(ctypes.byref(v1), ctypes.byref(v2), ctypes.byref(v3), ctypes.byref(e)) == 0
    print("e4m3 hw mismatches %d, block-scale mismatches %d, e2m1 bracket mismatches %d, rcp max rel %.3e"
          % (v1.value, v2.value, v3.value, e.value))
    assert v1.value == 0 and v2.value == 0 and v3.value == 0
    assert 0 < e.value < 2.0 ** -23
