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
