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


def test_training_step_graph_replay_matches_eager():
    """moe_forward then moe_backward (its gate branch forked onto the side
    stream and joined back) captured into one graph: replays reproduce the
    eager gradients bit for bit."""
    w = wl.Workload("graph_bwd", T=300, d=128, E=8, d_ff=256, k=2, cf=1.0, mode=wl.TOPK,
                    dtype="bf16", noisy=True)
    inp = wl.generate(w, seed=5, biases=True)
    d = to_device(w, inp)
    cfg = B.config_for(w)
    z = dict(device="cuda")
    dy = torch.from_numpy(wl.generate_dy(w, 5).view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.empty((w.T, w.d), dtype=torch.bfloat16, **z)
    out3 = torch.zeros(3, dtype=torch.float32, **z)
    ws = workspace(cfg)
    bws = torch.zeros(B.moe_backward_workspace_size(cfg), dtype=torch.uint8, **z)
    f = lambda *sh: torch.zeros(sh, dtype=torch.float32, **z)
    g = [torch.zeros((w.T, w.d), dtype=torch.bfloat16, **z), f(w.d, w.E), f(w.d, w.E), None,
         f(w.E, w.d, w.d_ff), f(w.E, w.d_ff), f(w.E, w.d_ff, w.d), f(w.E, w.d), f(w.T, w.k)]

    def step(stream):
        B.moe_forward(cfg, d["x"], d["Wg"], d["Wn"], d["noise"], None, d["W1"], d["b1"], d["W2"],
                      d["b2"], y, out3, ws, stream=stream)
        B.moe_backward(cfg, d["x"], d["Wg"], d["Wn"], d["noise"], d["W1"], d["W2"], d["b2"], None,
                       None, None, None, dy, 0.3, 0.3, 0.3, *g, ws, bws, stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s)  # eager, outside capture
    torch.cuda.synchronize()
    ref = [None if t is None else t.clone() for t in g]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(torch.cuda.current_stream())
    for t in g:
        if t is not None:
            t.zero_()
    torch.cuda.synchronize()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    st, det = B.moe_last_device_status(ws)
    assert st == 0, (B.STATUS_NAMES[st], det)
    for a, b in zip(g, ref):
        if a is not None:
            assert torch.equal(a, b), "graph replay gradient differs from the eager step"
