"""moe_forward under CUDA stream capture: the forward (with the balancing
finalize forked onto the library's side stream and joined back) is captured
into a graph on a non-default stream, replayed, and must reproduce an eager
call bit for bit."""
import numpy as np
import pytest
import torch

from gpu_harness import run_forward, to_device, workspace
from sparsely_gated_mixture_gb300 import binding as B
from sparsely_gated_mixture_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["noisy_top4_e16", "many_small_experts_e1024"])
def test_forward_graph_replay_matches_eager(name):
    w = wl.WORKLOADS[name].with_(T=700)
    inp = wl.generate(w, seed=21, biases=True)
    d = to_device(w, inp)
    ref = run_forward(w, d)
    assert ref["status"] == 0

    cfg = B.config_for(w)
    z = dict(device="cuda")
    y = torch.empty((w.T, w.d), dtype=torch.bfloat16, **z)
    out3 = torch.zeros(3, dtype=torch.float32, **z)
    idx = torch.empty((w.T, w.k), dtype=torch.int32, **z)
    gate = torch.empty((w.T, w.k), dtype=torch.float32, **z)
    pos = torch.empty((w.T, w.k), dtype=torch.int32, **z)
    keep = torch.empty((w.T, w.k), dtype=torch.uint8, **z)
    ws = workspace(cfg)

    def fwd(stream):
        B.moe_forward(cfg, d["x"], d["Wg"], d["Wn"], d["noise"], d["bias"], d["W1"], d["b1"],
                      d["W2"], d["b2"], y, out3, ws, idx, gate, pos, keep, stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fwd(s)  # outside capture: the library's one-time setup happens here
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fwd(torch.cuda.current_stream())
    y.zero_()
    out3.zero_()
    torch.cuda.synchronize()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    st, det = B.moe_last_device_status(ws)
    assert st == 0, (B.STATUS_NAMES[st], det)
    assert torch.equal(y, ref["y"]), "graph replay output differs from the eager forward"
    assert np.array_equal(out3.cpu().numpy(), ref["out3"])
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.array_equal(keep.cpu().numpy(), ref["keep"])
