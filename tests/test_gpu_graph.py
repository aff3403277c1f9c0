"""moe_expert_forward inside a CUDA graph: captured once on a stream, then
replayed on new inputs copied into the captured buffers; every replay
equals the eager forward bit for bit.  The small layers are launch-bound,
so graph replay is how a serving loop would run them."""
import numpy as np
import pytest

import nvfp4_w4a4_moe_top_gb300 as M
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from nvfp4_w4a4_moe_top_gb300 import build
    build.build()


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_forward_replays_in_a_cuda_graph(name):
    import torch
    from gpu_util import dev, host
    lay = synth.layer(name)
    T, E, k, d, F = lay.T, lay.E, lay.k, lay.d, lay.d_ff
    w1q, w2q = M.quantize_weights(dev(lay.w1())), M.quantize_weights(dev(lay.w2()))
    xd, lgd = dev(lay.x()), dev(lay.logits())
    out = torch.empty((T, d), dtype=torch.int16, device="cuda")
    ws = M.forward_workspace(T, E, k, d, F)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()

    def fwd(x, lg, o, w):
        M.moe_expert_forward(x, lg, T, E, k, d, F, w1q["codes"], w1q["sf"], w1q["g"], w2q["codes"], w2q["sf"],
                             w2q["g"], o, w, st)

    with torch.cuda.stream(s):  # first call outside the capture: device checks, attributes
        fwd(xd, lgd, out, ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fwd(xd, lgd, out, ws)
    ref_out = torch.empty_like(out)
    ref_ws = M.forward_workspace(T, E, k, d, F)
    for seed in [1, 2, 3]:
        other = synth.layer(name, seed=seed)
        xd.copy_(dev(other.x()))
        lgd.copy_(dev(other.logits()))
        g.replay()
        torch.cuda.synchronize()
        fwd(xd, lgd, ref_out, ref_ws)
        torch.cuda.synchronize()
        assert np.array_equal(host(out), host(ref_out)), seed
    assert int(st.item()) == 0
