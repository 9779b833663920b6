"""moe_dispatch_noalloc, the dispatch entry point for callers that cannot
allocate device memory (so cannot pass a workspace), against moe_dispatch on
the same gate outputs, twice in a row: its scratch is a static device array
that every call reuses and that keeps the previous call's contents.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_harness import to_device, workspace
from sparsely_gated_mixture_gb300 import binding as B
from sparsely_gated_mixture_gb300 import workloads as wl


def _outputs(w):
    T, k, E, A = w.T, w.k, w.E, w.T * w.k
    act = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    z = dict(device="cuda")
    return dict(pos=torch.full((T, k), -7, dtype=torch.int32, **z),
                keep=torch.full((T, k), 9, dtype=torch.uint8, **z),
                count=torch.full((E,), -7, dtype=torch.int32, **z),
                offset=torch.full((E + 1,), -7, dtype=torch.int32, **z),
                xbuf=torch.zeros((A, w.d), dtype=act, **z),
                row_token=torch.full((A,), -7, dtype=torch.int32, **z),
                row_gate=torch.zeros(A, dtype=torch.float32, **z))


def _same(ref, got):
    n = int(ref["offset"][-1].item())
    assert torch.equal(ref["pos"], got["pos"])
    assert torch.equal(ref["keep"], got["keep"])
    assert torch.equal(ref["count"], got["count"])
    assert torch.equal(ref["offset"], got["offset"])
    assert torch.equal(ref["xbuf"][:n], got["xbuf"][:n])
    assert torch.equal(ref["row_token"][:n], got["row_token"][:n])
    assert torch.equal(ref["row_gate"][:n], got["row_gate"][:n])


@pytest.mark.gpu
@pytest.mark.parametrize("w", [
    wl.WORKLOADS["noisy_top4_e16"].with_(T=517),
    wl.WORKLOADS["switch_top1_zipf_e64"].with_(T=900),
    wl.WORKLOADS["many_small_experts_e1024"].with_(T=1000),
], ids=lambda w: w.name)
def test_noalloc_dispatch_matches_dispatch_twice(w):
    inp = wl.generate(w, seed=21)
    d = to_device(w, inp)
    cfg = B.config_for(w)
    ws = workspace(cfg)
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    gate = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    thr = torch.empty((w.T, 2), dtype=torch.float32, device="cuda")
    B.moe_gate(cfg, d["x"], d["Wg"], d["Wn"], d["noise"], d["bias"], idx, gate, thr, ws)
    ref = _outputs(w)
    B.moe_dispatch(cfg, idx, gate, d["x"], ref["pos"], ref["keep"], ref["count"], ref["offset"],
                   ref["xbuf"], ref["row_token"], ref["row_gate"], ws)
    st, det = B.moe_last_device_status(ws)
    assert st == 0, (st, det)
    for _ in range(2):
        got = _outputs(w)
        B.moe_dispatch_noalloc(cfg, idx, gate, d["x"], got["pos"], got["keep"], got["count"],
                               got["offset"], got["xbuf"], got["row_token"], got["row_gate"])
        torch.cuda.synchronize()
        _same(ref, got)


@pytest.mark.gpu
def test_noalloc_dispatch_rejects_sizes_beyond_its_scratch():
    # 524288 assignments over 1024 experts need 8 MiB of histograms: more than 4 MiB.
    cfg = B.config(131072, 512, 1024, 1024, 4, 1.5)
    fake = 1 << 20  # never dereferenced: the size check fails first
    st = B.lib().moe_dispatch_noalloc(ctypes.byref(cfg), *([fake] * 10), None)
    assert st == 2  # MOE_ERR_UNSUPPORTED
    assert B.noalloc_scratch_need(cfg) > B.NOALLOC_SCRATCH_BYTES
    with pytest.raises(B.MoEError, match="static 4 MiB"):
        B.moe_dispatch_noalloc(cfg, *([fake] * 10), stream=0)
    # Too many experts is unsupported for another reason: no scratch message.
    wide = B.config(64, 64, 2048, 64, 2, 1.0)
    assert B.noalloc_scratch_need(wide) <= B.NOALLOC_SCRATCH_BYTES
    with pytest.raises(B.MoEError) as e:
        B.moe_dispatch_noalloc(wide, *([fake] * 10), stream=0)
    assert e.value.status == 2 and "scratch" not in str(e.value)


@pytest.mark.gpu
def test_noalloc_dispatch_reports_bad_expert_index():
    """An expert index outside [0, E) is skipped by every kernel of the call
    (pos = -1, keep = 0, no row) and recorded in the static array's status
    word, which moe_noalloc_last_status reads back and clears; the next call
    starts from a clear word. moe_dispatch, given the same indices, reports
    the same error through its workspace and writes the same outputs."""
    w = wl.WORKLOADS["noisy_top4_e16"].with_(T=300)
    inp = wl.generate(w, seed=22)
    d = to_device(w, inp)
    cfg = B.config_for(w)
    ws = workspace(cfg)
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    gate = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    thr = torch.empty((w.T, 2), dtype=torch.float32, device="cuda")
    B.moe_gate(cfg, d["x"], d["Wg"], d["Wn"], d["noise"], d["bias"], idx, gate, thr, ws)
    assert B.moe_last_device_status(ws)[0] == 0
    bad = idx.clone()
    bad[57, 2] = w.E  # flat index 57 * k + 2
    ref = _outputs(w)
    B.moe_dispatch(cfg, bad, gate, d["x"], ref["pos"], ref["keep"], ref["count"], ref["offset"],
                   ref["xbuf"], ref["row_token"], ref["row_gate"], ws)
    assert B.moe_last_device_status(ws) == (6, 57 * w.k + 2)
    got = _outputs(w)
    B.moe_dispatch_noalloc(cfg, bad, gate, d["x"], got["pos"], got["keep"], got["count"],
                           got["offset"], got["xbuf"], got["row_token"], got["row_gate"])
    assert B.moe_noalloc_last_status() == (6, 57 * w.k + 2)  # MOE_ERR_BOUNDS, flat index
    assert B.moe_noalloc_last_status() == (0, 0)  # read once, then cleared
    _same(ref, got)
    assert int(got["pos"][57, 2].item()) == -1 and int(got["keep"][57, 2].item()) == 0
    good = _outputs(w)
    B.moe_dispatch_noalloc(cfg, idx, gate, d["x"], good["pos"], good["keep"], good["count"],
                           good["offset"], good["xbuf"], good["row_token"], good["row_gate"])
    assert B.moe_noalloc_last_status() == (0, 0)
