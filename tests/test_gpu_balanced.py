"""GPU parity of strictly balanced gating (moe_forward_balanced) against the
fp64 oracle: the batchwise mask (exact, or explained near-ties at an expert's
m-th place), the layer output and L_batchwise."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import (FLOOR_SIGMAS, TIE_TOL, act_to_f64, check_close, dev_act, dev_f32,
                         f32_output_floor, router_value_err)
from sparsely_gated_mixture_gb300 import binding as B
from sparsely_gated_mixture_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _unpack(bits, E):
    T, W = bits.shape
    out = np.zeros((T, W * 32), np.uint8)
    for w in range(W):
        for b in range(32):
            out[:, w * 32 + b] = (bits[:, w] >> np.uint32(b)) & np.uint32(1)
    return out[:, :E]


def reconcile_mask(P, ref_mask, gpu_mask, m, tol=TIE_TOL):
    """Columns where the GPU's picks differ from the oracle's must differ only
    among tokens whose oracle P lies within tol of the column's m-th value.
    Returns (mask to use, differing columns, unexplained columns)."""
    diff = np.nonzero((ref_mask != gpu_mask).any(axis=0))[0]
    bad = []
    for i in diff:
        mth = -np.sort(-P[:, i])[m - 1]
        rows = np.nonzero(ref_mask[:, i] != gpu_mask[:, i])[0]
        if gpu_mask[:, i].sum() != m or np.any(np.abs(P[rows, i] - mth) > tol * max(1.0, mth)):
            bad.append(int(i))
    return gpu_mask if len(diff) else ref_mask, [int(i) for i in diff], bad


def check_balanced(w, inp, tokens, thr_seed=None):
    cfg = B.config_for(w)
    dev = "cuda"
    act = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    x = dev_act(inp["x"], w.dtype)
    Wg, bias = dev_f32(inp["Wg"]), dev_f32(inp["bias"])
    W1, b1 = dev_act(inp["W1"], w.dtype), dev_act(inp["b1"], w.dtype)
    W2, b2 = dev_act(inp["W2"], w.dtype), dev_act(inp["b2"], w.dtype)
    ref = oracle.bal_forward(dict(inp, mode_bal=0), tokens=tokens)
    m, P = ref["m"], ref["P"]
    thr = None
    if thr_seed is not None:  # near each column's m-th value, so some tokens disagree
        srt = -np.sort(-P, axis=0)
        jitter = np.random.default_rng(thr_seed).integers(-3, 4, size=w.E)
        thr = np.array([srt[min(max(m - 1 + j, 0), w.T - 1), i] * 0.999
                        for i, j in enumerate(jitter)], np.float32)
    y = torch.empty((w.T, w.d), dtype=act, device=dev)
    loss = torch.zeros(1, dtype=torch.float32, device=dev) if thr is not None else None
    W = (w.E + 31) // 32
    bits = torch.zeros((w.T, W), dtype=torch.int32, device=dev)
    ws = torch.zeros(B.moe_balanced_workspace_size(cfg), dtype=torch.uint8, device=dev)
    B.moe_forward_balanced(cfg, x, Wg, bias, None if thr is None else dev_f32(thr), W1, b1, W2,
                           b2, y, loss, bits, ws)
    st, det = B.moe_last_device_status(ws)
    assert st == 0, (B.STATUS_NAMES[st], det)
    gmask = _unpack(bits.cpu().numpy().view(np.uint32), w.E)
    assert np.all(gmask.sum(axis=0) == m), "an expert did not get exactly m tokens"
    used, cols, bad = reconcile_mask(P, ref["mask"], gmask, m)
    assert not bad, f"batchwise mask differs beyond near-ties in experts {bad[:10]}"
    z = (P * used).sum(axis=1, keepdims=True)
    gate = np.where(used == 1, P / np.where(z > 0, z, 1.0), 0.0)
    idx = np.tile(np.arange(w.E, dtype=np.int32), (w.T, 1))
    y_ref, badf = oracle.layer_out(inp["x"], idx, gate, used, inp["W1"], inp["W2"], inp["b1"],
                                   inp["b2"], tokens)
    assert not badf
    yg = act_to_f64(y[torch.as_tensor(tokens, device=dev).long()])
    floor = None
    if w.dtype == "f32":
        # The gates are P renormalised over the token's picks, P = Softmax(H):
        # each H error moves P's relative value by at most twice it, and the
        # renormalisation doubles that again.
        allc = np.tile(np.arange(w.E), (w.T, 1))
        eh = router_value_err(inp["x"], inp["Wg"], None, None, inp["bias"], allc)
        g_rel = 4.0 * FLOOR_SIGMAS * float(eh.max())
        floor = f32_output_floor(inp["x"][tokens], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                                 idx[tokens], gate[tokens], used[tokens], g_rel)
    err = check_close(yg, y_ref, w.dtype, "balanced layer output", floor)
    if thr is not None:
        # L_batchwise sums differences P - T_i with T_i close to P, so it
        # inherits the fp32 router's error in P (about 1e-6 relative, from
        # logits accurate to ~1e-6 absolute) amplified by P / |P - T_i|. The
        # bound: the 1e-4 rule on the terms, plus a relative error of 1e-5 in P
        # on every term that is nonzero or could flip (|P - T_i| within it).
        want = oracle.bal_loss(P, used, thr)
        th = thr.astype(np.float64)[None, :]
        ind = (P > th).astype(np.float64) - used
        terms = np.abs(ind * (P - th)).sum()
        live = (ind != 0) | (np.abs(P - th) <= 1e-5 * P)
        got = float(loss.cpu().numpy()[0])
        lim = 1e-4 * terms + 1e-5 * P[live].sum() + 1e-9
        assert abs(got - want) <= lim, (got, want, terms, lim)
    return dict(tie_cols=cols, y_err=err, unpicked=int((used.sum(axis=1) == 0).sum()))


def _w(name, T, d, E, d_ff, k, dtype="bf16"):
    return wl.Workload(name, T=T, d=d, E=E, d_ff=d_ff, k=k, cf=1.0, mode=wl.TOPK, dtype=dtype,
                       noisy=False)


SMALL = {
    "bal_e8_k2": _w("bal_e8_k2", 333, 128, 8, 64, 2),
    "bal_e16_k4": _w("bal_e16_k4", 400, 64, 16, 128, 4),
    "bal_e64_k1": _w("bal_e64_k1", 1000, 64, 64, 64, 1),
    "bal_k_equals_E": _w("bal_k_equals_E", 130, 64, 4, 64, 4),
    "bal_ragged_f32": _w("bal_ragged_f32", 129, 36, 7, 50, 2, dtype="f32"),
    "bal_e40_d72": _w("bal_e40_d72", 300, 72, 40, 64, 3),
    # edge cases: one token (m = 1), m = 1 with many tokens, a ragged tail
    # of the 1024-token select chunks, more than 32 experts per mask word set
    "bal_single_token": _w("bal_single_token", 1, 64, 4, 64, 2),
    "bal_m1": _w("bal_m1", 100, 64, 64, 64, 1),
    "bal_ragged_chunks": _w("bal_ragged_chunks", 2049, 64, 8, 64, 2),
    "bal_e100_k8": _w("bal_e100_k8", 400, 64, 100, 64, 8),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_balanced_small_parity(name):
    w = SMALL[name]
    inp = wl.generate(w, seed=89, biases=True)
    inp["bias"] = (np.random.default_rng(2).standard_normal(w.E) * 0.3).astype(np.float32)
    check_balanced(w, inp, np.arange(w.T, dtype=np.int32), thr_seed=5)


def test_balanced_exact_ties():
    """A zero router with a coarse bias: every token has the same P row, so
    every column is one long tie and the first m tokens must be taken."""
    w = _w("bal_ties", 200, 64, 8, 64, 2)
    inp = wl.generate(w, seed=91)
    inp["Wg"] = np.zeros_like(inp["Wg"])
    inp["bias"] = np.round(np.random.default_rng(4).standard_normal(w.E)).astype(np.float32)
    rep = check_balanced(w, inp, np.arange(w.T, dtype=np.int32))
    assert not rep["tie_cols"]


@pytest.mark.parametrize("name", sorted(wl.BAL_WORKLOADS))
def test_balanced_full_size_sampled(name):
    w = wl.BAL_WORKLOADS[name]
    inp = wl.generate(w, seed=0)
    rng = np.random.default_rng(6)
    tokens = np.array(sorted(set(rng.choice(w.T, 128, replace=False).tolist()) | {0, w.T - 1}),
                      np.int32)
    rep = check_balanced(w, inp, tokens, thr_seed=7)
    print(name, "tie columns:", len(rep["tie_cols"]), "tokens no expert took:", rep["unpicked"],
          "y max err:", rep["y_err"])
