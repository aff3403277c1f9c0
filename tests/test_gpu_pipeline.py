"""The pipelined forward on host-resident batches (moe_pipeline_*): every
step's host output equals moe_expert_forward of the same batch bit for bit,
with several different batches in flight (depth 2 and 3), on small layers
and on the 64k-token layer."""
import numpy as np
import pytest

import nvfp4_w4a4_moe_top_gb300 as M
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from nvfp4_w4a4_moe_top_gb300 import build
    build.build()


def pinned(a):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).pin_memory()


def direct(lay, x, lg, w1q, w2q):
    import torch
    from gpu_util import dev, host
    T, E, k, d, F = x.shape[0], lay.E, lay.k, lay.d, lay.d_ff
    out = torch.empty((T, d), dtype=torch.int16, device="cuda")
    ws = M.forward_workspace(T, E, k, d, F)
    M.moe_expert_forward(dev(x), dev(lg), T, E, k, d, F, w1q["codes"], w1q["sf"], w1q["g"], w2q["codes"], w2q["sf"],
                         w2q["g"], out, ws)
    torch.cuda.synchronize()
    return host(out, np.uint16)


@pytest.mark.parametrize("name,depth,steps", [("tiny", 2, 5), ("small", 3, 7), ("qwen64k", 2, 3)])
def test_pipeline_equals_direct_forward(name, depth, steps):
    import torch
    from gpu_util import dev
    lay = synth.layer(name)
    T, E, k, d, F = lay.T, lay.E, lay.k, lay.d, lay.d_ff
    w1q, w2q = M.quantize_weights(dev(lay.w1())), M.quantize_weights(dev(lay.w2()))
    nb = min(steps, 3)
    batches = [(synth.layer(name, seed=s).x(), synth.layer(name, seed=s).logits()) for s in range(nb)]
    xs = [pinned(b[0]) for b in batches]
    ls = [pinned(b[1]) for b in batches]
    outs = [torch.full((T, d), 0x5A5A, dtype=torch.int16).pin_memory() for _ in range(steps)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pipe = M.Pipeline(T, E, k, d, F, depth=depth)
    try:
        for i in range(steps):
            pipe.submit(xs[i % nb], ls[i % nb], outs[i], w1q, w2q, st)
        pipe.synchronize()
    finally:
        pipe.close()
    assert int(st.item()) == 0
    ref = [direct(lay, b[0], b[1], w1q, w2q) for b in batches]
    for i in range(steps):
        assert np.array_equal(outs[i].numpy().view(np.uint16), ref[i % nb]), i
