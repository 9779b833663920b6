"""The library's expert-parallel calls on one GPU (moe_expert_counts,
moe_dispatch_ranked, moe_expert_ffn on received rows, moe_combine,
moe_aux_totals, moe_aux_from_totals), with two ranks run in turn and the
exchange done by slicing on the device, against the oracle's forward over the
whole batch; and ep_forward through LibraryOps on a one-rank process group.
Ranks run one after another: no kernel of one waits for another's."""
import socket

import numpy as np
import pytest
import torch

import oracle
from gpu_harness import (act_to_f64, check_close, check_gate_rel, check_rel, oracle_gate,
                         reconcile_selection, to_device)
from sparsely_gated_mixture_gb300 import binding as B
from sparsely_gated_mixture_gb300 import expert_parallel as EP
from sparsely_gated_mixture_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _rank_inputs(d, lo, hi):
    sub = dict(d)
    sub["x"] = d["x"][lo:hi].contiguous()
    sub["noise"] = None if d["noise"] is None else d["noise"][lo:hi].contiguous()
    return sub


@pytest.mark.parametrize("splits,cf", [([0, 257, 600], 0.9), ([0, 300, 600], 1.25),
                                       ([0, 100, 350, 600], 0.7)])
def test_ranked_dispatch_emulated_ranks(splits, cf):
    W = len(splits) - 1
    w = wl.Workload("ep_gpu", T=600, d=128, E=12 if W == 3 else 8, d_ff=256, k=2, cf=cf,
                    mode=wl.TOPK, dtype="bf16", noisy=True)
    E = w.E
    inp = wl.generate(w, seed=61, biases=True)
    d = to_device(w, inp)
    C = oracle.capacity(w.T, E, w.k, w.cf, w.min_cap)
    z = dict(device="cuda")
    ranks = []
    for r in range(W):
        lo, hi = splits[r], splits[r + 1]
        cfg = B.config(hi - lo, w.d, E, w.d_ff, w.k, w.cf)
        ws = torch.zeros(B.moe_workspace_size(cfg), dtype=torch.uint8, **z)
        sub = _rank_inputs(d, lo, hi)
        idx = torch.empty((hi - lo, w.k), dtype=torch.int32, **z)
        gate = torch.empty((hi - lo, w.k), dtype=torch.float32, **z)
        thr = torch.empty((hi - lo, 2), dtype=torch.float32, **z)
        B.moe_gate(cfg, sub["x"], sub["Wg"], sub["Wn"], sub["noise"], sub["bias"], idx, gate, thr,
                   ws)
        counts = torch.empty(E, dtype=torch.int32, **z)
        B.moe_expert_counts(cfg, idx, counts, ws)
        ranks.append(dict(cfg=cfg, ws=ws, sub=sub, idx=idx, gate=gate, counts=counts))
    counts_all = torch.stack([rk["counts"] for rk in ranks]).contiguous()
    for rk in ranks:  # the counts are the selection's choices per expert
        assert torch.equal(rk["counts"], torch.bincount(rk["idx"].long().flatten(),
                                                        minlength=E).to(torch.int32))
    for r, rk in enumerate(ranks):
        c = rk["cfg"]
        A = c.T * c.k
        rk.update(pos=torch.empty((c.T, c.k), dtype=torch.int32, **z),
                  keep=torch.empty((c.T, c.k), dtype=torch.uint8, **z),
                  count=torch.empty(E, dtype=torch.int32, **z),
                  offset=torch.empty(E + 1, dtype=torch.int32, **z),
                  xbuf=torch.empty((A, w.d), dtype=torch.bfloat16, **z),
                  row_token=torch.empty(A, dtype=torch.int32, **z),
                  row_gate=torch.empty(A, dtype=torch.float32, **z))
        B.moe_dispatch_ranked(c, C, counts_all, W, r, rk["idx"], rk["gate"], rk["sub"]["x"],
                              rk["pos"], rk["keep"], rk["count"], rk["offset"], rk["xbuf"],
                              rk["row_token"], rk["row_gate"], rk["ws"])
    # The choices against the oracle's (near-ties reconciled), then slots and
    # drops against the single-batch rule applied to the choices used.
    ref_gate = oracle_gate(inp)
    gpu_idx = np.concatenate([rk["idx"].cpu().numpy() for rk in ranks])
    used, ties, bad = reconcile_selection(ref_gate["H"], ref_gate["idx"], gpu_idx)
    assert not bad
    pos_ref, keep_ref, _ = oracle.slots(used, E, C)
    base = np.zeros(E, np.int64)
    for r, rk in enumerate(ranks):
        lo, hi = splits[r], splits[r + 1]
        iv = rk["idx"].cpu().numpy()
        assert np.array_equal(rk["pos"].cpu().numpy() + base[iv], pos_ref[lo:hi])
        assert np.array_equal(rk["keep"].cpu().numpy(), keep_ref[lo:hi])
        base += rk["counts"].cpu().numpy()
    # The exchange: rank q holds experts q*E/W ..; each source's rows for them
    # are one contiguous range of its packed buffer.
    n_loc = E // W
    ffn_out = [torch.zeros((rk["cfg"].T * w.k, w.d), dtype=torch.float32, **z) for rk in ranks]
    for q in range(W):
        e0, e1 = q * n_loc, (q + 1) * n_loc
        for r, rk in enumerate(ranks):
            off = rk["offset"].cpu().tolist()
            a, b = off[e0], off[e1]
            if a == b:
                continue
            rows = rk["xbuf"][a:b].contiguous()
            offs = torch.tensor([o - a for o in off[e0:e1 + 1]], dtype=torch.int32, **z)
            lc = B.config(b - a, w.d, n_loc, w.d_ff, 1, float(n_loc))
            hb = torch.empty((b - a, w.d_ff), dtype=torch.bfloat16, **z)
            zb = torch.empty((b - a, w.d), dtype=torch.float32, **z)
            lws = torch.zeros(B.moe_workspace_size(lc), dtype=torch.uint8, **z)
            B.moe_expert_ffn(lc, rows, offs, rk["row_gate"][a:b].clone(), d["W1"][e0:e1],
                             d["b1"][e0:e1], d["W2"][e0:e1], d["b2"][e0:e1], hb, zb, lws)
            ffn_out[r][a:b] = zb
    ys, totals = [], torch.zeros((4, E), dtype=torch.float32, **z)
    for r, rk in enumerate(ranks):
        y = torch.empty_like(rk["sub"]["x"])
        B.moe_combine(rk["cfg"], rk["sub"]["x"], ffn_out[r], rk["pos"], rk["keep"], rk["idx"],
                      rk["offset"], y, rk["ws"])
        ys.append(y)
        t = torch.empty((4, E), dtype=torch.float32, **z)
        B.moe_aux_totals(rk["cfg"], rk["ws"], t)
        totals += t
        st, det = B.moe_last_device_status(rk["ws"])
        assert st == 0, (B.STATUS_NAMES[st], det)
    out3 = torch.empty(3, dtype=torch.float32, **z)
    B.moe_aux_from_totals(ranks[0]["cfg"], w.T, totals, out3, ranks[0]["ws"])
    # Outputs and losses of the whole batch.
    g_ref = oracle.gates_given(ref_gate["H"], used, 0)
    gpu_gate = np.concatenate([rk["gate"].cpu().numpy() for rk in ranks])
    check_gate_rel(gpu_gate, g_ref)
    y_ref, badf = oracle.layer_out(inp["x"], used, g_ref, keep_ref, inp["W1"], inp["W2"],
                                   inp["b1"], inp["b2"], np.arange(w.T, dtype=np.int32))
    assert not badf
    check_close(act_to_f64(torch.cat(ys)), y_ref, "bf16", "expert-parallel output")
    ax = oracle.aux(ref_gate["c"], ref_gate["sigma"], ref_gate["H"], used, g_ref,
                    ref_gate["hk"], ref_gate["hk1"], True)
    check_rel(out3.cpu().numpy(), ax["out3"], "whole-batch balancing losses")


def test_ep_forward_library_ops_one_rank():
    """ep_forward with LibraryOps on a one-rank NCCL group: the module's
    glue around the C ABI (buffers, offsets, alignment) against moe_forward
    on the same inputs."""
    import torch.distributed as dist

    w = wl.Workload("ep_one", T=333, d=128, E=8, d_ff=256, k=2, cf=0.9, mode=wl.TOPK,
                    dtype="bf16", noisy=True)
    inp = wl.generate(w, seed=62, biases=True)
    d = to_device(w, inp)
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    store = dist.TCPStore("127.0.0.1", port, 1, True)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    try:
        cfg = B.config_for(w)
        ws = torch.zeros(B.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
        ops = EP.LibraryOps(cfg, ws)
        y, out3, info = EP.ep_forward(ops, d["x"], d["Wg"], d["Wn"], d["noise"], d["bias"],
                                      d["W1"], d["b1"], d["W2"], d["b2"], E=w.E, k=w.k, cf=w.cf)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    st, det = B.moe_last_device_status(ws)
    assert st == 0, (B.STATUS_NAMES[st], det)
    y2 = torch.empty_like(y)
    out3b = torch.zeros(3, dtype=torch.float32, device="cuda")
    ws2 = torch.zeros(B.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    B.moe_forward(cfg, d["x"], d["Wg"], d["Wn"], d["noise"], d["bias"], d["W1"], d["b1"],
                  d["W2"], d["b2"], y2, out3b, ws2)
    assert B.moe_last_device_status(ws2)[0] == 0
    # moe_forward may keep the expert outputs in bf16 (one more rounding per term)
    check_close(act_to_f64(y), act_to_f64(y2), "bf16", "ep_forward against moe_forward")
    check_rel(out3.cpu().numpy(), out3b.cpu().numpy(), "balancing losses")
