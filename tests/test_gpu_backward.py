"""The backward through the C ABI (moe_backward, moe_gate_backward) against
the fp64 oracle's backward (oracle.backward).

Tolerances, derived from the arithmetic (the oracle is exact):

* The GPU's expert path holds three bf16 operands the oracle keeps exact: the
  forward's h rows, the gate-scaled dy rows (g * dy) and dpre. Each rounding
  is within 2^-9 relative, products are exact in fp32, sums are fp32. So every
  expert-side gradient entry, a sum of terms each carrying at most two such
  roundings, is within 2^-8 * (sum of |terms|) of the exact value: the test
  allows 1e-2 * (sum of |terms|), with the sums of |terms| formed in numpy
  from exact fp64 quantities. fp32 layers (the CUDA-core path, fp32 row
  buffers) round nothing to bf16: 1e-4 * (sum of |terms|).
* ReLU pattern: the GPU decides h > 0 on its fp32 pre-activation. Where the
  exact pre-activation is within 1e-5 of its own magnitude scale
  (sum_i |x_i W1_if| + |b1_f|) of zero the two sides may disagree; such
  entries' terms are allowed in full.
* dL/dgate of a kept choice, <dy, U> = <dy W2^T, h> + <dy, b2>, inherits h's
  rounding: within 1e-2 * sum_f |D_f h_f| (+ fp32 terms).
* The router gradients are fp32 computations of exact-to-fp32 inputs, except
  for what they inherit from dL/dgate: through the top-k softmax Jacobian,
  |d dH_S_j| <= G_j (eps_j + sum_l G_l eps_l); through the Switch softmax,
  |d dH_e| <= p_e ([e = e0] + p_e0) eps_0; then into dc, into sigma through
  the noise and into z through sigmoid(z). Those bounds are carried to dW_g,
  dW_noise, the bias and dx. Fed the oracle's own dL/dgate (the stage call
  moe_gate_backward), the router gradients are within 1e-4 of their sums of
  |terms| plus 1e-4 of the largest entry.
* dx is bf16: one more rounding (2^-9 relative, allowed 4e-3 * |ref|).
* Besides the elementwise bounds, every weight gradient's Frobenius error is
  within 2e-2 of its norm (statistical: the roundings are independent).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_harness import dev_act, reconcile_selection, to_device, workspace
from sparsely_gated_mixture_gb300 import binding as B
from sparsely_gated_mixture_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

W = wl.Workload
CASES = {
    # noisy top-2 with capacity drops, all three losses, biases
    "noisy_top2_e8": (W("noisy_top2_e8", T=256, d=128, E=8, d_ff=256, k=2, cf=1.0, mode=wl.TOPK,
                        dtype="bf16", noisy=True), (0.5, 0.7, 0.3)),
    # clean Switch top-1 with the Zipf router bias: the full-softmax path
    "switch_clean_e4": (W("switch_clean_e4", T=192, d=64, E=4, d_ff=128, k=1, cf=1.0,
                          mode=wl.SWITCH, dtype="bf16", noisy=False, zipf_bias=True),
                        (0.2, 0.0, 0.9)),
    # widths that leave partial 128-row / 256-column tiles, a ragged T
    "noisy_top4_e16_ragged": (W("noisy_top4_e16_ragged", T=300, d=192, E=16, d_ff=320, k=4,
                                cf=2.0, mode=wl.TOPK, dtype="bf16", noisy=True), (0.4, 0.6, 0.0)),
    # k = E: every expert always chosen, no load gradient
    "noisy_k_eq_E": (W("noisy_k_eq_E", T=128, d=64, E=4, d_ff=128, k=4, cf=1.0, mode=wl.TOPK,
                       dtype="bf16", noisy=True), (0.3, 0.5, 0.2)),
    # capacity 1 with 64 experts: most experts get no row at all
    "sparse_e64_cap1": (W("sparse_e64_cap1", T=64, d=64, E=64, d_ff=128, k=1, cf=1.0,
                          mode=wl.TOPK, dtype="bf16", noisy=True), (0.5, 0.5, 0.5)),
    # the CUDA-core expert backward: the fp32 Switch toy, a noisy fp32 top-2,
    # and bf16 widths that are not multiples of 64
    "switch_toy_f32": (wl.WORKLOADS["switch_top1_toy"], (0.2, 0.0, 0.5)),
    "noisy_top2_f32": (W("noisy_top2_f32", T=200, d=48, E=6, d_ff=80, k=2, cf=1.0, mode=wl.TOPK,
                         dtype="f32", noisy=True), (0.5, 0.5, 0.5)),
    "bf16_widths_96_160": (W("bf16_widths_96_160", T=160, d=96, E=4, d_ff=160, k=2, cf=1.0,
                             mode=wl.TOPK, dtype="bf16", noisy=True), (0.4, 0.4, 0.4)),
}
# Cases whose expert backward runs on the CUDA cores (no kernel variants).
SIMT = {"switch_toy_f32", "noisy_top2_f32", "bf16_widths_96_160"}


def _bf(a):
    """Exact fp64 values of a bf16 (uint16 bits) or fp32 array."""
    if a.dtype == np.uint16:
        return wl.bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


def _rel(w):
    """Per-term rounding allowance: bf16 operands (h, g*dy, dpre) or fp32 only."""
    return 1e-2 if w.dtype == "bf16" else 1e-4


def _f32(t):
    return t.float().cpu().numpy().astype(np.float64)


def _gpu(w, inp, dy_bits, weights, big_to_host=True):
    """moe_forward then moe_backward; returns host arrays (the weight
    gradients stay on the device only when big_to_host is False) and the
    device outputs under "dev"."""
    d = to_device(w, inp)
    cfg = B.config_for(w)
    T, k, E, dd, dff = w.T, w.k, w.E, w.d, w.d_ff
    dev = "cuda"
    act = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    y = torch.empty((T, dd), dtype=act, device=dev)
    out3 = torch.zeros(3, dtype=torch.float32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gate = torch.empty((T, k), dtype=torch.float32, device=dev)
    pos = torch.empty((T, k), dtype=torch.int32, device=dev)
    keep = torch.empty((T, k), dtype=torch.uint8, device=dev)
    ws = workspace(cfg)
    B.moe_forward(cfg, d["x"], d["Wg"], d["Wn"], d["noise"], d["bias"], d["W1"], d["b1"], d["W2"],
                  d["b2"], y, out3, ws, idx, gate, pos, keep)
    st, det = B.moe_last_device_status(ws)
    assert st == 0, (st, det)
    bws = torch.zeros(B.moe_backward_workspace_size(cfg), dtype=torch.uint8, device=dev)
    dy = dev_act(dy_bits, w.dtype)
    f = lambda *s: torch.full(s, float("nan"), dtype=torch.float32, device=dev)
    o = dict(dx=torch.empty((T, dd), dtype=act, device=dev), dWg=f(dd, E),
             dWn=f(dd, E) if w.noisy else None, dbias=f(E) if inp["bias"] is not None else None,
             dW1=f(E, dd, dff), db1=f(E, dff), dW2=f(E, dff, dd), db2=f(E, dd), dgate=f(T, k))
    B.moe_backward(cfg, d["x"], d["Wg"], d["Wn"], d["noise"], d["W1"], d["W2"], d["b2"], idx, gate,
                   pos, keep, dy, *weights, o["dx"], o["dWg"], o["dWn"], o["dbias"], o["dW1"],
                   o["db1"], o["dW2"], o["db2"], o["dgate"], ws, bws)
    st, det = B.moe_last_device_status(ws)
    assert st == 0, (st, det)
    # The gate's share alone, from given dL/dgate (the caller passes the oracle's).
    def gate_stage(dgate_in, wl_, wa_):
        g = dict(dWg=f(dd, E), dWn=f(dd, E) if w.noisy else None,
                 dbias=f(E) if inp["bias"] is not None else None, dxg=f(T, dd))
        B.moe_gate_backward(cfg, d["x"], d["Wg"], d["Wn"], d["noise"], idx, gate,
                            torch.from_numpy(dgate_in.astype(np.float32)).to(dev), wl_, wa_,
                            g["dWg"], g["dWn"], g["dbias"], g["dxg"], ws, bws)
        s2, d2 = B.moe_last_device_status(ws)
        assert s2 == 0, (s2, d2)
        return {n: (None if v is None else _f32(v)) for n, v in g.items()}
    big = ("dW1", "dW2")
    host = {n: (None if v is None or (n in big and not big_to_host) else _f32(v))
            for n, v in o.items()}
    host.update(idx=idx.cpu().numpy(), keep=keep.cpu().numpy(), gate=gate.cpu().numpy(),
                gate_stage=gate_stage, dev=o)
    return host


def _bounds(w, inp, dy, fw, ref):
    """Sums of |terms| for every expert-side gradient, the ambiguous-ReLU
    allowances and the dL/dgate error bound eps [T,k] (see the module doc)."""
    T, k, E, d, dff = w.T, w.k, w.E, w.d, w.d_ff
    R = _rel(w)
    X = _bf(inp["x"])
    W1, W2 = _bf(inp["W1"]), _bf(inp["W2"])
    b1 = _bf(inp["b1"]) if inp["b1"] is not None else np.zeros((E, dff))
    b2 = _bf(inp["b2"]) if inp["b2"] is not None else np.zeros((E, d))
    idx, keep, gate = fw["idx"], fw["keep"], fw["gate"]
    bW2, bdb2 = np.zeros((E, dff, d)), np.zeros((E, d))
    bW1, bdb1 = np.zeros((E, d, dff)), np.zeros((E, dff))
    bx = np.zeros((T, d))
    eps = np.zeros((T, k))
    for e in range(E):
        tj = np.argwhere((idx == e) & (keep == 1))
        if tj.size == 0:
            continue
        ts, js = tj[:, 0], tj[:, 1]
        g = gate[ts, js][:, None]
        Xe, Ye = X[ts], dy[ts]
        pre = Xe @ W1[e] + b1[e]
        scale = np.abs(Xe) @ np.abs(W1[e]) + np.abs(b1[e])
        amb = np.abs(pre) <= 1e-5 * scale
        h = np.maximum(pre, 0.0)
        D = Ye @ W2[e].T
        dh = g * D
        mask = pre > 0
        bW2[e] = R * (np.abs(h).T @ np.abs(g * Ye))
        bdb2[e] = 1e-4 * np.abs(g * Ye).sum(0)
        bW1[e] = R * (np.abs(Xe).T @ np.abs(dh * mask)) + np.abs(Xe).T @ np.abs(dh * amb)
        bdb1[e] = R * np.abs(dh * mask).sum(0) + np.abs(dh * amb).sum(0)
        part = R * (np.abs(dh * mask) @ np.abs(W1[e]).T) + np.abs(dh * amb) @ np.abs(W1[e]).T
        np.add.at(bx, ts, part)
        eps[ts, js] = R * np.abs(D * h).sum(1) + 1e-4 * np.abs(Ye * b2[e]).sum(1)
    eps += 1e-4 * np.abs(ref["dgate"]) + 1e-4 * np.abs(ref["dgate"]).max() + 1e-7
    return dict(dW2=bW2, db2=bdb2, dW1=bW1, db1=bdb1, bx=bx, eps=eps)


def _router_bounds(w, inp, fw, eps):
    """Bounds on dc [T,E] and dz [T,E] inherited from dL/dgate errors eps."""
    T, k, E = w.T, w.k, w.E
    H = fw["H"]
    Bdc = np.zeros((T, E))
    if w.mode == wl.SWITCH:
        p = np.exp(H - H.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        e0 = fw["idx"][:, 0]
        p0 = p[np.arange(T), e0]
        Bdc = p * p0[:, None] * eps[:, :1]
        Bdc[np.arange(T), e0] += p0 * eps[:, 0]
    else:
        G = fw["gate"]
        tot = (G * eps).sum(1)
        for j in range(k):
            Bdc[np.arange(T), fw["idx"][:, j]] += G[:, j] * (eps[:, j] + tot)
    Bdz = np.zeros((T, E))
    if w.noisy:
        sig = -np.expm1(-fw["sigma"])
        Bdz = np.abs(inp["noise"].astype(np.float64)) * sig * Bdc
    return Bdc, Bdz


def _check(got, ref, lim, what, norm=True):
    err = np.abs(got - ref)
    bad = err > lim
    if bad.any():
        i = np.unravel_index(np.argmax(err - lim), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} entries out of bound; worst at {i}: "
                             f"got {got[i]:.6g} ref {ref[i]:.6g} bound {lim[i]:.3g}")
    if norm:
        nr = np.linalg.norm(ref)
        assert np.linalg.norm(got - ref) <= 2e-2 * nr + 1e-6, (what, np.linalg.norm(got - ref), nr)


@pytest.mark.parametrize("variant", ["auto", "single", "pair", "pair_k_backwards"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_backward_matches_oracle(name, variant, monkeypatch):
    """variant: the expert GEMMs' kernel as the library picks it, or forced
    to the one-CTA or the CTA-pair form; pair_k_backwards also makes every
    CTA-pair tile walk K from its last block (by default only the odd waves
    of tiles do, which these small layers never reach)."""
    if variant != "auto":
        if name in SIMT:
            pytest.skip("the CUDA-core expert backward has one form")
        monkeypatch.setenv("MOE_BWD_TC_VARIANT", variant.split("_")[0])
        if variant == "pair_k_backwards":
            monkeypatch.setenv("MOE_FFN_SNAKE", "all")
    w, weights = CASES[name]
    seed = 11
    inp = wl.generate(w, seed=seed, biases=True)
    if inp["bias"] is None:  # (the Switch case keeps its Zipf bias)
        inp["bias"] = np.random.default_rng(seed).normal(0.0, 0.3, w.E).astype(np.float32)
    dy_bits = wl.generate_dy(w, seed)
    dy = _bf(dy_bits)
    fw = oracle.forward(inp)
    ref = oracle.backward(inp, dy, *weights)
    gpu = _gpu(w, inp, dy_bits, weights)
    used, ties, bad = reconcile_selection(fw["H"], fw["idx"], gpu["idx"])
    assert not bad and not ties, f"selection differs (ties {ties}, unexplained {bad}): reseed"
    assert np.array_equal(gpu["keep"], fw["keep"])
    b = _bounds(w, inp, dy, fw, ref)
    _check(gpu["dgate"], ref["dgate"], b["eps"], "dgate", norm=False)
    for n in ("dW2", "db2", "dW1", "db1"):
        _check(gpu[n], ref[n], b[n] + 1e-6, n)
    # Experts that received no row have zero weight gradients.
    empty = [e for e in range(w.E) if not ((fw["idx"] == e) & (fw["keep"] == 1)).any()]
    for e in empty:
        assert np.all(gpu["dW1"][e] == 0) and np.all(gpu["dW2"][e] == 0), e
    Bdc, Bdz = _router_bounds(w, inp, fw, b["eps"])
    X = np.abs(_bf(inp["x"]))
    Wg, Wn = np.abs(inp["Wg"].astype(np.float64)), None
    fl = lambda a: 1e-4 * np.abs(a).max() + 1e-7
    _check(gpu["dWg"], ref["dWg"], X.T @ Bdc + 1e-4 * (X.T @ np.abs(ref["dc"])) + fl(ref["dWg"]),
           "dWg")
    rx = Bdc @ Wg.T + 1e-4 * (np.abs(ref["dc"]) @ Wg.T)
    if w.noisy:
        Wn = np.abs(inp["Wn"].astype(np.float64))
        _check(gpu["dWn"], ref["dWn"],
               X.T @ Bdz + 1e-4 * (X.T @ np.abs(ref["dz"])) + fl(ref["dWn"]), "dWn")
        rx += Bdz @ Wn.T + 1e-4 * (np.abs(ref["dz"]) @ Wn.T)
    _check(gpu["dbias"], ref["dbias"],
           Bdc.sum(0) + 1e-4 * np.abs(ref["dc"]).sum(0) + fl(ref["dbias"]), "dbias")
    out_round = 4e-3 if w.dtype == "bf16" else 1e-6  # dx is stored in act_dtype
    _check(gpu["dx"], ref["dx"], b["bx"] + rx + out_round * np.abs(ref["dx"]) + 1e-5, "dx",
           norm=False)
    # The gate's share alone, from the oracle's dL/dgate: fp32 against fp64.
    gs = gpu["gate_stage"](ref["dgate"], weights[1], weights[2])
    _check(gs["dWg"], ref["dWg"], 1e-4 * (X.T @ np.abs(ref["dc"])) + fl(ref["dWg"]), "stage dWg")
    _check(gs["dbias"], ref["dbias"], 1e-4 * np.abs(ref["dc"]).sum(0) + fl(ref["dbias"]),
           "stage dbias")
    gx = np.abs(ref["dc"]) @ Wg.T
    if w.noisy:
        _check(gs["dWn"], ref["dWn"], 1e-4 * (X.T @ np.abs(ref["dz"])) + fl(ref["dWn"]),
               "stage dWn")
        gx += np.abs(ref["dz"]) @ Wn.T
    dxg_ref = ref["dc"] @ inp["Wg"].astype(np.float64).T
    if w.noisy:
        dxg_ref += ref["dz"] @ inp["Wn"].astype(np.float64).T
    _check(gs["dxg"], dxg_ref, 1e-4 * gx + fl(dxg_ref), "stage dx_gate")


def test_backward_repeatable():
    """Two backward calls on one forward give identical bits (fixed-order
    sums, no floating-point atomics)."""
    w, weights = CASES["noisy_top2_e8"]
    inp = wl.generate(w, seed=3, biases=True)
    inp["bias"] = np.random.default_rng(3).normal(0.0, 0.3, w.E).astype(np.float32)
    dy_bits = wl.generate_dy(w, 3)
    a = _gpu(w, inp, dy_bits, weights)
    b = _gpu(w, inp, dy_bits, weights)
    for n in ("dx", "dWg", "dWn", "dbias", "dW1", "db1", "dW2", "db2", "dgate"):
        assert np.array_equal(a[n], b[n]), n


def test_backward_full_size_properties():
    """The large-expert layer (T = 8192, d = 4096, E = 8, d_ff = 14336, top-2)
    at full size, where the oracle's whole backward is out of reach, through
    facts that hold at any size:

    * expert e's output is linear in (W2, b2) and positively homogeneous in
      (W1, b1), so sum over its kept rows of g_r * dL/dgate_r (w_importance
      = 0) equals both <dW2, W2> + <db2, b2> and <dW1, W1> + <db1, b1> +
      sum_r g_r <dy_t, b2>; allowed 1e-2 of the sums of |terms| (torch fp32
      on the device, |h| |W2| |dy| and |h| |dy W2^T|);
    * a common shift of a token's logits changes nothing: the bias gradient
      and every row of dW_g sum to zero (1e-3 of the sums of magnitudes);
    * dL/dgate of sampled kept choices equals <dy_t, E_e(x_t)> from the oracle
      (one expert at a time), within the bound of the small cases."""
    w = wl.WORKLOADS["top2_large_experts"]
    weights = (0.0, 0.5, 0.5)
    inp = wl.generate(w, seed=0, biases=True)
    inp["bias"] = np.random.default_rng(0).normal(0.0, 0.3, w.E).astype(np.float32)
    dy_bits = wl.generate_dy(w, 0)
    gpu = _gpu(w, inp, dy_bits, weights, big_to_host=False)
    T, k, E, d, dff = w.T, w.k, w.E, w.d, w.d_ff
    dev = "cuda"
    tb = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    X, DY = tb(inp["x"]).float(), tb(dy_bits).float()
    W1, W2 = tb(inp["W1"]), tb(inp["W2"])
    b1, b2 = tb(inp["b1"]).float(), tb(inp["b2"]).float()
    dW1, dW2 = gpu["dev"]["dW1"], gpu["dev"]["dW2"]
    db1, db2 = gpu["dev"]["db1"], gpu["dev"]["db2"]
    idx, keep = gpu["idx"], gpu["keep"]
    for e in range(E):
        tj = np.argwhere((idx == e) & (keep == 1))
        ts = torch.from_numpy(tj[:, 0]).to(dev)
        # the gates the GPU forward used, and its dL/dgate
        g = torch.from_numpy(gpu["gate"][tj[:, 0], tj[:, 1]].astype(np.float64)).to(dev)
        dg = torch.from_numpy(gpu["dgate"][tj[:, 0], tj[:, 1]]).to(dev)
        lhs = float((g * dg).sum())
        w2e, w1e = W2[e].float(), W1[e].float()
        rhs2 = float((dW2[e].double() * w2e.double()).sum() + (db2[e].double() * b2[e].double()).sum())
        yb = float((g * (DY[ts].double() @ b2[e].double())).sum())
        rhs1 = float((dW1[e].double() * w1e.double()).sum() + (db1[e].double() * b1[e].double()).sum()) + yb
        h = torch.relu(X[ts] @ w1e + b1[e])
        Dm = DY[ts] @ w2e.T
        m2 = float((g.abs().float()[:, None] * (h.abs() @ w2e.abs()) * DY[ts].abs()).sum())
        m1 = float((g.abs().float()[:, None] * h.abs() * Dm.abs()).sum())
        assert abs(lhs - rhs2) <= 1e-2 * m2 + 1e-3, (e, lhs, rhs2, m2)
        assert abs(lhs - rhs1) <= 1e-2 * (m1 + m2) + 1e-3, (e, lhs, rhs1, m1)
    db = gpu["dbias"]
    assert abs(db.sum()) <= 1e-3 * np.abs(db).sum()
    rows = gpu["dWg"].sum(1)
    assert np.abs(rows).max() <= 1e-3 * np.abs(gpu["dWg"]).sum(1).max()
    # Sampled dL/dgate against the oracle, one expert at a time.
    rng = np.random.default_rng(5)
    kept = np.argwhere(keep == 1)
    X64, DY64 = _bf(inp["x"]), _bf(dy_bits)
    W1h, W2h = _bf(inp["W1"]), _bf(inp["W2"])
    b1h, b2h = _bf(inp["b1"]), _bf(inp["b2"])
    for t, j in kept[rng.choice(len(kept), 6, replace=False)]:
        e = int(idx[t, j])
        one = np.full((T, 1), e, np.int32)
        yv, _ = oracle.layer_out(inp["x"], one, np.ones((T, 1)), np.ones((T, 1), np.uint8),
                                 inp["W1"], inp["W2"], inp["b1"], inp["b2"],
                                 tokens=np.array([t], np.int32))
        U = yv[0] - X64[t]
        want = float(DY64[t] @ U)
        pre = X64[t] @ W1h[e] + b1h[e]
        bound = 1e-2 * float(np.abs((DY64[t] @ W2h[e].T) * np.maximum(pre, 0)).sum()) + \
            1e-4 * float(np.abs(DY64[t] * b2h[e]).sum()) + 1e-4 * abs(want) + 1e-6
        assert abs(gpu["dgate"][t, j] - want) <= bound, (t, j, gpu["dgate"][t, j], want, bound)


def test_backward_full_size_sampled_entries():
    """The large-expert layer at full size (T = 8192, d = 4096, E = 8, d_ff =
    14336, top-2), as bench.py --backward runs it: sampled entries of dW1,
    dW2, db1 and db2 against the oracle's entry-by-entry sums over each
    expert's kept rows, within 1e-2 of each entry's sum of |terms| (the bf16
    rounding of h, g*dy and dpre), once the GPU's routing equals the oracle's."""
    w = wl.WORKLOADS["top2_large_experts"]
    weights = (0.01, 0.01, 0.01)
    inp = wl.generate(w, seed=0, biases=True)
    dy_bits = wl.generate_dy(w, 0)
    gpu = _gpu(w, inp, dy_bits, weights, big_to_host=False)
    fw = oracle.forward(inp, tokens=np.zeros(1, np.int32))
    used, ties, bad = reconcile_selection(fw["H"], fw["idx"], gpu["idx"])
    assert not bad and not ties, f"routing differs (ties {ties}, unexplained {bad})"
    assert np.array_equal(gpu["keep"], fw["keep"])
    rng = np.random.default_rng(7)
    entries = []
    for e in range(w.E):
        entries += [("dW1", e, int(rng.integers(w.d)), int(rng.integers(w.d_ff))),
                    ("dW2", e, int(rng.integers(w.d_ff)), int(rng.integers(w.d))),
                    ("db1", e, int(rng.integers(w.d_ff)), 0), ("db2", e, int(rng.integers(w.d)), 0)]
    want, absum = oracle.backward_entries(inp, _bf(dy_bits), entries)
    dev = gpu["dev"]
    for (kind, e, a, b), v, m in zip(entries, want, absum):
        t = dev[kind]
        got = float(t[e, a, b] if kind in ("dW1", "dW2") else t[e, a])
        assert abs(got - v) <= 1e-2 * m + 1e-6, (kind, e, a, b, got, v, m)
