"""Helpers for the GPU parity tests: host <-> device copies of the numpy
arrays the oracle uses (no method arithmetic)."""
import os
import subprocess

import numpy as np
import pytest

torch = pytest.importorskip("torch")


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host(t, dtype=None):
    a = t.detach().cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


def zeros(shape, dtype, guard=0):
    return torch.zeros(shape, dtype=dtype, device="cuda")


def f32_of_bf16(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    n = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (n if n > 0 else 1.0)


def build_test_so(name):
    root = os.path.dirname(os.path.abspath(__file__))
    src = os.path.join(root, "gpu_src", name + ".cu")
    out_dir = os.path.join(root, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "lib%s.so" % name)
    csrc = os.path.join(os.path.dirname(root), "nvfp4_w4a4_moe_top_gb300", "csrc")
    deps = [src] + [os.path.join(csrc, f) for f in os.listdir(csrc) if f.endswith(".cuh")]
    if not os.path.exists(so) or os.path.getmtime(so) < max(os.path.getmtime(d) for d in deps):
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-Xcompiler", "-fPIC", "-shared", src, "-o", so], check=True)
    return so
