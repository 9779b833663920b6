"""Helpers for the GPU parity tests: move generated inputs to the device, run
the library through its C ABI, and compare with the oracle under the rules:

* expert indices, slot positions, drop masks, counts and offsets bit-exact,
  except tokens whose oracle margin between the k-th and (k+1)-th noisy logit
  (or, for an order swap inside the top k, between the swapped logits) is
  below TIE_TOL; such tokens are reported, and the GPU's choice is then fed to
  the oracle for everything downstream;
* bf16 outputs within 2e-2 * (1 + |ref|); fp32 outputs, gates, gate
  thresholds and balancing losses within 1e-4 relative.

Near zero a relative bound asks for more than fp32 arithmetic can give (a
value that cancels to 1e-6 carries the rounding error of its much larger
terms). So fp32 outputs and gate thresholds are checked against
max(1e-4 |ref|, F): F is an estimate of the fp32 evaluation's own rounding
error, built from the computation (``f32_output_floor``,
``router_value_err``), and it exceeds 1e-4 |ref| only for values near zero.
Gates have no floor: every gate is a positive softmax value.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from sparsely_gated_mixture_gb300 import binding as B
from sparsely_gated_mixture_gb300 import workloads as wl

TIE_TOL = 1e-6
BF16_TOL = 2e-2
F32_RTOL = 1e-4
U32 = 2.0 ** -24  # unit roundoff of fp32 (round to nearest)
FLOOR_SIGMAS = 6.0  # floors are this many estimated standard deviations


# ----------------------------------------------------------------------------- fp32 error floors
# A sum s = a_1 + ... + a_n evaluated in fp32 incurs one rounding per
# addition, |delta_i| <= u, on the partial sum S_i = a_1 + ... + a_i, so
# fl(s) - s = sum_i delta_i S_i to first order. Treating the roundings as
# independent and of mean zero (Higham and Mary, "A New Approach to
# Probabilistic Rounding Error Analysis", SIAM J. Sci. Comput. 2019) its
# standard deviation is at most u * sqrt(sum_i S_i^2). Products and bias adds
# contribute their own u-relative terms; errors of a sum's inputs pass
# through it weighted by their coefficients. FLOOR_SIGMAS such deviations
# make the floor. The partial sums are taken in the oracle's index order; the
# GPU's blocked order has partial sums of the same size.


def _sum_var(terms: np.ndarray, axis: int) -> np.ndarray:
    """u^2 * (sum_i S_i^2 + sum_i a_i^2): the additions' and the products'
    rounding variance of the sum of ``terms`` along ``axis``."""
    S = np.cumsum(terms, axis=axis)
    return U32 ** 2 * ((S * S).sum(axis=axis) + (terms * terms).sum(axis=axis))


def router_value_err(x: np.ndarray, Wg, Wn, noise, bias, cols: np.ndarray) -> np.ndarray:
    """Standard deviation estimate of the fp32 router's error in H[t, e] for
    e = cols[t, q]: c = x Wg + b (one sum over d), sigma = Softplus(x Wn)
    (a sum, then a few-ulp Softplus whose slope is sigmoid(z) <= 1),
    H = c + n sigma."""
    T = x.shape[0]
    out = np.empty(cols.shape, np.float64)
    Wg = np.asarray(Wg, np.float64)
    for q in range(cols.shape[1]):
        e = cols[:, q]
        tg = x * Wg[:, e].T  # [T, d]
        c = tg.sum(axis=1) + (0.0 if bias is None else np.asarray(bias, np.float64)[e])
        var = _sum_var(tg, 1) + U32 ** 2 * c * c
        if Wn is not None:
            tn = x * np.asarray(Wn, np.float64)[:, e].T
            z = tn.sum(axis=1)
            sg = np.logaddexp(0.0, z)
            slope = 1.0 / (1.0 + np.exp(-z))
            n = np.asarray(noise, np.float64)[np.arange(T), e]
            var_s = slope ** 2 * _sum_var(tn, 1) + (4 * U32 * sg) ** 2
            H = c + n * sg
            var = var + n * n * var_s + U32 ** 2 * ((n * sg) ** 2 + H * H)
        out[:, q] = np.sqrt(var)
    return out


def f32_output_floor(x, W1, b1, W2, b2, experts, gates, keep, g_rel):
    """FLOOR_SIGMAS times the estimated standard deviation of the fp32 layer
    output's error, per element of y [n, d] for the token rows x [n, d]:
    pre = x W1[e] + b1[e] (a sum over d), h = ReLU(pre) (1-Lipschitz),
    o = h W2[e] + b2[e] (a sum over d_ff, carrying h's error through W2),
    z = g o (g with relative error g_rel: the gate's own error), and
    y = x + z_1 + ... in choice order (kept choices only)."""
    x = np.asarray(x, np.float64)
    n, d = x.shape
    var_y = np.zeros((n, d))
    S = x.copy()
    for j in range(experts.shape[1]):
        live = keep[:, j].astype(bool) & (experts[:, j] >= 0)
        if not live.any():
            continue
        rows = np.nonzero(live)[0]
        e = experts[rows, j]
        xs = x[rows]
        W1e = np.asarray(W1, np.float64)[e]            # [m, d, d_ff]
        terms = xs[:, :, None] * W1e
        pre = terms.sum(axis=1)
        if b1 is not None:
            pre = pre + np.asarray(b1, np.float64)[e]
        var_pre = _sum_var(terms, 1) + U32 ** 2 * pre * pre
        h = np.maximum(pre, 0.0)
        W2e = np.asarray(W2, np.float64)[e]            # [m, d_ff, d]
        terms2 = h[:, :, None] * W2e
        o = terms2.sum(axis=1)
        if b2 is not None:
            o = o + np.asarray(b2, np.float64)[e]
        var_o = (np.einsum("mf,mfd->md", var_pre, W2e * W2e) + _sum_var(terms2, 1)
                 + U32 ** 2 * o * o)
        g = np.asarray(gates, np.float64)[rows, j][:, None]
        z = g * o
        var_z = g * g * var_o + (g_rel ** 2 + U32 ** 2) * z * z
        S[rows] += z
        var_y[rows] += var_z + U32 ** 2 * S[rows] ** 2
    return FLOOR_SIGMAS * np.sqrt(var_y)


def dev_act(a, dtype: str):
    if a is None:
        return None
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def dev_f32(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def to_device(w: wl.Workload, inp: dict) -> dict:
    dt = w.dtype
    return dict(x=dev_act(inp["x"], dt), Wg=dev_f32(inp["Wg"]), Wn=dev_f32(inp["Wn"]),
                noise=dev_f32(inp["noise"]), bias=dev_f32(inp["bias"]), W1=dev_act(inp["W1"], dt),
                b1=dev_act(inp["b1"], dt), W2=dev_act(inp["W2"], dt), b2=dev_act(inp["b2"], dt))


def act_to_f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def act_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy()
    return t.view(torch.int32).cpu().numpy()


def workspace(cfg) -> torch.Tensor:
    return torch.zeros(B.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")


def run_forward(w, d, aux=True, keep_outputs=True):
    """moe_forward through the C ABI. Returns a dict of host arrays."""
    cfg = B.config_for(w)
    T, k, E = w.T, w.k, w.E
    act = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    y = torch.empty((T, w.d), dtype=act, device="cuda")
    out3 = torch.zeros(3, dtype=torch.float32, device="cuda") if aux else None
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    pos = torch.empty((T, k), dtype=torch.int32, device="cuda")
    keep = torch.empty((T, k), dtype=torch.uint8, device="cuda")
    ws = workspace(cfg)
    B.moe_forward(cfg, d["x"], d["Wg"], d["Wn"], d["noise"], d["bias"], d["W1"], d["b1"], d["W2"],
                  d["b2"], y, out3, ws, idx, gate, pos, keep)
    st, det = B.moe_last_device_status(ws)
    return dict(status=st, detail=det, y=y, out3=None if out3 is None else out3.cpu().numpy(),
                idx=idx.cpu().numpy(), gate=gate.cpu().numpy(), pos=pos.cpu().numpy(),
                keep=keep.cpu().numpy(), ws=ws)


def run_stages(w, d):
    """The five stage entry points in turn, keeping every intermediate."""
    cfg = B.config_for(w)
    T, k, E = w.T, w.k, w.E
    A = T * k
    act = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    z = dict(device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, **z)
    gate = torch.empty((T, k), dtype=torch.float32, **z)
    thr = torch.empty((T, 2), dtype=torch.float32, **z)
    ws = workspace(cfg)
    B.moe_gate(cfg, d["x"], d["Wg"], d["Wn"], d["noise"], d["bias"], idx, gate, thr, ws)
    pos = torch.empty((T, k), dtype=torch.int32, **z)
    keep = torch.empty((T, k), dtype=torch.uint8, **z)
    count = torch.empty(E, dtype=torch.int32, **z)
    offset = torch.empty(E + 1, dtype=torch.int32, **z)
    xbuf = torch.empty((A, w.d), dtype=act, **z)
    row_token = torch.full((A,), -1, dtype=torch.int32, **z)
    row_gate = torch.empty(A, dtype=torch.float32, **z)
    B.moe_dispatch(cfg, idx, gate, d["x"], pos, keep, count, offset, xbuf, row_token, row_gate, ws)
    hbuf = torch.empty((A, w.d_ff), dtype=act, **z)
    zbuf = torch.empty((A, w.d), dtype=torch.float32, **z)
    B.moe_expert_ffn(cfg, xbuf, offset, row_gate, d["W1"], d["b1"], d["W2"], d["b2"], hbuf, zbuf, ws)
    y = torch.empty((T, w.d), dtype=act, **z)
    B.moe_combine(cfg, d["x"], zbuf, pos, keep, idx, offset, y, ws)
    out3 = torch.zeros(3, dtype=torch.float32, **z)
    imp = torch.zeros(E, dtype=torch.float32, **z)
    load = torch.zeros(E, dtype=torch.float32, **z)
    B.moe_aux_loss(cfg, ws, out3, imp, load)
    st, det = B.moe_last_device_status(ws)
    h = lambda t: t.cpu().numpy()
    return dict(status=st, detail=det, idx=h(idx), gate=h(gate), thr=h(thr), pos=h(pos),
                keep=h(keep), count=h(count), offset=h(offset), xbuf=xbuf, row_token=h(row_token),
                row_gate=h(row_gate), hbuf=hbuf, zbuf=zbuf, y=y, out3=h(out3), importance=h(imp),
                load=h(load))


def oracle_gate(inp):
    c, s, H, bad = oracle.router(inp["x"], inp["Wg"], inp["Wn"], inp["noise"], inp["bias"])
    idx, gate, hk, hk1 = oracle.select(H, int(inp["k"]), int(inp["mode"]))
    return dict(c=c, sigma=s, H=H, idx=idx, gate=gate, hk=hk, hk1=hk1, nonfinite=bad)


def reconcile_selection(H, ref_idx, gpu_idx, tol=TIE_TOL):
    """Tokens where the GPU's expert list differs from the oracle's. Each must
    be explained by a near-tie: the GPU's list, read in the oracle's fp64 H,
    must be non-increasing within tol and no unchosen expert may beat its last
    entry by more than tol. Returns (idx to use downstream, list of tokens,
    list of unexplained tokens)."""
    diff = np.nonzero((ref_idx != gpu_idx).any(axis=1))[0]
    used = ref_idx.copy()
    ties, bad = [], []
    E = H.shape[1]
    for t in diff:
        g = gpu_idx[t]
        ok = bool(np.all((g >= 0) & (g < E))) and len(set(g.tolist())) == len(g)
        if ok:
            hv = H[t, g]
            ok = bool(np.all(np.diff(hv) <= tol))
            rest = np.setdiff1d(np.arange(E), g)
            if ok and rest.size:
                ok = bool(H[t, rest].max() <= hv.min() + tol)
        (ties if ok else bad).append(int(t))
        if ok:
            used[t] = g
    return used, ties, bad


def check_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str, floor=None):
    """bf16: |err| <= 2e-2 (1 + |ref|). fp32: |err| <= max(1e-4 |ref|, floor),
    the floor an fp32 rounding-error estimate (required for fp32)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if dtype == "bf16":
        lim = BF16_TOL * (1.0 + np.abs(ref))
    else:
        assert floor is not None, "fp32 checks need the rounding-error floor"
        lim = np.maximum(F32_RTOL * np.abs(ref), floor)
        FLOOR_USE.append((what, int((floor > F32_RTOL * np.abs(ref)).sum()), int(ref.size)))
    err = np.abs(got - ref)
    worst = np.unravel_index(np.argmax(err - lim), err.shape) if err.size else None
    assert np.all(err <= lim), (f"{what}: max err {err.max():.3e} at {worst}, "
                                f"got {got[worst]:.6g} ref {ref[worst]:.6g}")
    return float(err.max()) if err.size else 0.0


FLOOR_USE = []  # (what, elements whose bound is the floor, elements checked)


def check_gate_rel(got, ref, what="gate"):
    """Gates: pure relative 1e-4 (every compared gate is a positive softmax
    value). Returns the largest relative error, for the output floor."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(ref > 0), f"{what}: a reference gate is not positive"
    rel = np.abs(got - ref) / ref
    assert np.all(rel <= F32_RTOL), f"{what}: max relative err {rel.max():.3e}"
    return float(rel.max()) if rel.size else 0.0


def check_rel(got, ref, what, rtol=F32_RTOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    lim = rtol * np.maximum(np.abs(ref), 1e-30)
    assert np.all(err <= lim), f"{what}: got {got} ref {ref}"


# ----------------------------------------------------------------------------- hierarchical layer


def hier_to_device(w, inp: dict) -> dict:
    dt = w.dtype
    return dict(x=dev_act(inp["x"], dt), Wp=dev_f32(inp["Wp"]), Wpn=dev_f32(inp["Wpn"]),
                noise_p=dev_f32(inp["noise_p"]), Ws=dev_f32(inp["Ws"]), Wsn=dev_f32(inp["Wsn"]),
                noise_s=dev_f32(inp["noise_s"]), W1=dev_act(inp["W1"], dt),
                b1=dev_act(inp["b1"], dt), W2=dev_act(inp["W2"], dt), b2=dev_act(inp["b2"], dt))


def run_hier_forward(w, d, aux=True):
    """moe_forward_hier through the C ABI. Returns host arrays (y on device)."""
    cfg = B.hier_config_for(w)
    T, k = w.T, w.k
    act = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    y = torch.empty((T, w.d), dtype=act, device="cuda")
    out2 = torch.zeros(2, dtype=torch.float32, device="cuda") if aux else None
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    pos = torch.empty((T, k), dtype=torch.int32, device="cuda")
    keep = torch.empty((T, k), dtype=torch.uint8, device="cuda")
    ws = torch.zeros(B.moe_hier_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    B.moe_forward_hier(cfg, d["x"], d["Wp"], d["Wpn"], d["noise_p"], d["Ws"], d["Wsn"],
                       d["noise_s"], d["W1"], d["b1"], d["W2"], d["b2"], y, out2, ws, idx, gate,
                       pos, keep)
    st, det = B.moe_last_device_status(ws)
    return dict(status=st, detail=det, y=y, out2=None if out2 is None else out2.cpu().numpy(),
                idx=idx.cpu().numpy(), gate=gate.cpu().numpy(), pos=pos.cpu().numpy(),
                keep=keep.cpu().numpy())


def _group_rows(Hs, groups, b):
    """Hs[t, groups[t]*b .. groups[t]*b + b - 1] for every t: [T, b]."""
    T = Hs.shape[0]
    cols = groups[:, None].astype(np.int64) * b + np.arange(b)[None, :]
    return Hs[np.arange(T)[:, None], cols]


def reconcile_hier(ref, gpu_idx, a, b, kp, ks, tol=TIE_TOL):
    """The GPU's flat choices against the oracle's, level by level: its
    primary list (idx // b every ks choices) must match or be a near-tie in
    the oracle's fp64 primary logits, and in each picked group its secondary
    list must match the oracle's selection in that group or be a near-tie in
    the oracle's secondary logits. Returns (choices to use downstream, tied
    tokens, unexplained tokens)."""
    T = gpu_idx.shape[0]
    idx_p_gpu = (gpu_idx[:, ::ks] // b).astype(np.int32)
    used_p, ties_p, bad_p = reconcile_selection(ref["Hp"], ref["idx_p"], idx_p_gpu, tol)
    used = np.empty_like(gpu_idx)
    ties, bad = set(ties_p), set(bad_p)
    for q in range(kp):
        groups = used_p[:, q]
        sub = _group_rows(ref["Hs"], groups, b)
        own, _, _, _ = oracle.select(sub, ks, oracle.TOPK_SOFTMAX)
        loc = gpu_idx[:, q * ks:(q + 1) * ks] - groups[:, None] * b
        u, t_s, b_s = reconcile_selection(sub, own, loc.astype(np.int32), tol)
        used[:, q * ks:(q + 1) * ks] = u + groups[:, None] * b
        ties |= set(t_s)
        bad |= set(b_s)
    return used.astype(np.int32), sorted(ties), sorted(bad)


def hier_given(inp, ref, used, w, tokens):
    """The oracle's gates, slots, output rows and hierarchical losses for the
    flat choices ``used`` (its own where the GPU agreed)."""
    a, b, kp, ks = w.a, w.b, w.kp, w.ks
    T, E, k = w.T, w.E, w.k
    idx_p = (used[:, ::ks] // b).astype(np.int32)
    g_p = oracle.gates_given(ref["Hp"], idx_p, oracle.TOPK_SOFTMAX)
    _, _, hkp, hk1p = oracle.select(ref["Hp"], kp, oracle.TOPK_SOFTMAX)
    load_p = oracle.aux(ref["cp"], ref["sp"], ref["Hp"], idx_p, g_p, hkp, hk1p,
                        inp["Wpn"] is not None)["load"]
    gate = np.empty((T, k), np.float64)
    hks = np.empty((T, kp), np.float64)
    hk1s = np.empty((T, kp), np.float64)
    for q in range(kp):
        sub = _group_rows(ref["Hs"], idx_p[:, q], b)
        loc = (used[:, q * ks:(q + 1) * ks] - idx_p[:, q:q + 1] * b).astype(np.int32)
        gate[:, q * ks:(q + 1) * ks] = g_p[:, q:q + 1] * oracle.gates_given(
            sub, loc, oracle.TOPK_SOFTMAX)
        _, _, hks[:, q], hk1s[:, q] = oracle.select(sub, ks, oracle.TOPK_SOFTMAX)
    hx = oracle.hier_aux(idx_p, ref["cs"], ref["ss"], used, gate, hks, hk1s, load_p, a, b, ks,
                         inp["Wsn"] is not None)
    C = oracle.capacity(T, E, k, w.cf, w.min_cap)
    pos, keep, _ = oracle.slots(used, E, C)
    y, bad = oracle.layer_out(inp["x"], used, gate, keep, inp["W1"], inp["W2"], inp["b1"],
                              inp["b2"], tokens)
    assert not bad
    return dict(gate=gate, pos=pos, keep=keep, y=y, **hx)
