"""Pins of the fp64 oracle to facts the pages and mathematics fix.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError if
that oracle disagrees with:

* numbers printed on the pages (``tests/golden/lesson_worked_examples.json``),
* closed forms (capacity, Switch auxiliary loss under uniform and collapsed
  routing, zero initialisation),
* independent library routines (numpy matmul / einsum / sort, scipy's normal
  CDF) on small inputs, and
* brute force (a Monte-Carlo redraw of one expert's noise for P(x,i)).

``test_oracle_pins.py`` runs them on the oracle; ``test_oracle_mutations.py``
runs them on copies of the oracle with planted mistakes and checks that every
mistake fails at least one pin.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
from scipy.special import ndtr

from sparsely_gated_mixture_gb300.workloads import bf16_bits_to_f32, f32_to_bf16_bits

TOPK, SWITCH = 0, 1
_GOLDEN_PATH = os.path.join(os.path.dirname(__file__), "golden", "lesson_worked_examples.json")
with open(_GOLDEN_PATH) as _f:
    GOLDEN = json.load(_f)


def _dense_gates(idx, gate, E):
    T, k = idx.shape
    G = np.zeros((T, E))
    for t in range(T):
        for j in range(k):
            G[t, idx[t, j]] = gate[t, j]
    return G


def _router_for_H(clean, H):
    """Router inputs whose noisy logits are H: d = E + 1, x = [clean, 1],
    W_g = [I; 0] and W_noise = [0; ln(e - 1)], so sigma = Softplus(ln(e-1)) = 1
    and noise = H - clean."""
    E = len(clean)
    x = np.array([list(clean) + [1.0]], np.float32)
    Wg = np.zeros((E + 1, E), np.float32)
    Wg[:E, :E] = np.eye(E, dtype=np.float32)
    Wn = np.zeros((E + 1, E), np.float32)
    Wn[E, :] = math.log(math.e - 1.0)
    noise = (np.asarray(H, np.float64) - np.asarray(clean, np.float64)).astype(np.float32)[None]
    return x, Wg, Wn, noise


def _ref_order(h, k):
    """Experts ordered by (H descending, index ascending), first k."""
    return sorted(range(len(h)), key=lambda e: (-h[e], e))[:k]


def _x64(x):
    return bf16_bits_to_f32(x).astype(np.float64) if x.dtype == np.uint16 else x.astype(np.float64)


def _ffn_all(X, W1, b1, W2, b2):
    """E_e(X) for every expert e with numpy matmuls: [E, T, d]."""
    E = W1.shape[0]
    out = []
    for e in range(E):
        h = X @ _x64(W1[e]) + (0.0 if b1 is None else _x64(b1[e]))
        h = np.maximum(h, 0.0)
        out.append(h @ _x64(W2[e]) + (0.0 if b2 is None else _x64(b2[e])))
    return np.stack(out)


# ----------------------------------------------------------------------------- gating


def pin_lesson_gates(orc):
    """The lesson's four-expert worked examples, routed through the router."""
    for ex in GOLDEN["gating"]:
        x, Wg, Wn, noise = _router_for_H(ex["clean"], ex["H"])
        c, s, H, bad = orc.router(x, Wg, Wn, noise)
        assert not bad
        np.testing.assert_allclose(c[0], ex["clean"], atol=1e-12)
        np.testing.assert_allclose(s[0], 1.0, atol=1e-6)
        np.testing.assert_allclose(H[0], ex["H"], atol=1e-6)
        idx, gate, _, _ = orc.select(H, ex["k"], TOPK)
        G = _dense_gates(idx, gate, 4)[0]
        np.testing.assert_allclose(G, ex["gates"], atol=ex["tol"] + 1e-12, err_msg=ex["source"])
        assert np.count_nonzero(G) == ex["k"]
        assert abs(G.sum() - 1.0) < 1e-12


def pin_lesson_second_draw(orc):
    ex = GOLDEN["second_draw"]
    H = np.array([[1.4, 0.2, 1.5, -1.0]])  # only 1.5 and 1.4 are printed; the rest are lower
    idx, gate, _, _ = orc.select(H, ex["k"], TOPK)
    assert list(idx[0]) == ex["top2_experts"]
    np.testing.assert_allclose(gate[0], ex["gates"], atol=ex["tol"])


def pin_zero_init(orc):
    """W_g = W_noise = 0: clean logits 0, sigma = Softplus(0) = log 2, H = noise*log 2."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 7)).astype(np.float32)
    noise = rng.standard_normal((5, 4)).astype(np.float32)
    z = np.zeros((7, 4), np.float32)
    c, s, H, _ = orc.router(x, z, z, noise)
    assert np.all(c == 0.0)
    np.testing.assert_allclose(s, math.log(2.0), rtol=1e-15)
    ex = GOLDEN["zero_init"]
    assert abs(s[0, 0] - ex["sigma"]) < ex["tol"]
    np.testing.assert_allclose(H, noise.astype(np.float64) * math.log(2.0), rtol=1e-15)


def pin_router_numpy(orc):
    """Router against numpy's fp64 matmul, with bias and noise, fp32 and bf16 x."""
    rng = np.random.default_rng(2)
    T, d, E = 7, 13, 5
    x32 = rng.standard_normal((T, d)).astype(np.float32)
    Wg = (rng.standard_normal((d, E)) / math.sqrt(d)).astype(np.float32)
    Wn = (rng.standard_normal((d, E)) / math.sqrt(d)).astype(np.float32)
    noise = rng.standard_normal((T, E)).astype(np.float32)
    bias = rng.standard_normal(E).astype(np.float32)
    for x in (x32, f32_to_bf16_bits(x32)):
        X = _x64(x)
        c_ref = X @ Wg.astype(np.float64) + bias.astype(np.float64)
        s_ref = np.logaddexp(0.0, X @ Wn.astype(np.float64))
        H_ref = c_ref + noise.astype(np.float64) * s_ref
        c, s, H, _ = orc.router(x, Wg, Wn, noise, bias)
        np.testing.assert_allclose(c, c_ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(s, s_ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(H, H_ref, rtol=1e-12, atol=1e-12)
        c0, s0, H0, _ = orc.router(x, Wg)
        np.testing.assert_allclose(c0, X @ Wg.astype(np.float64), rtol=1e-12, atol=1e-12)
        assert np.all(s0 == 0.0) and np.all(H0 == c0)


def pin_select_bruteforce(orc):
    """Top-k order with ties (lower index first), gates, thresholds; Switch."""
    rng = np.random.default_rng(3)
    T, E = 60, 6
    H = np.round(rng.standard_normal((T, E)), 1)  # one decimal: many exact ties
    H[0] = 0.5  # a row of all-equal logits
    for k in range(1, E + 1):
        idx, gate, hk, hk1 = orc.select(H, k, TOPK)
        for t in range(T):
            order = _ref_order(list(H[t]), E)
            assert list(idx[t]) == order[:k], (k, t)
            w = np.exp(H[t, order[:k]] - H[t, order[0]])
            np.testing.assert_allclose(gate[t], w / w.sum(), rtol=1e-13)
            assert hk[t] == H[t, order[k - 1]]
            assert hk1[t] == (H[t, order[k]] if k < E else -np.inf)
        G = _dense_gates(idx, gate, E)
        assert np.all(np.count_nonzero(G, axis=1) == k)
        np.testing.assert_allclose(G.sum(axis=1), 1.0, rtol=1e-13)
    idx, gate, _, _ = orc.select(H, 1, SWITCH)
    p = np.exp(H - H.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    am = np.argmax(H, axis=1)  # numpy: first index on ties
    assert np.array_equal(idx[:, 0], am)
    np.testing.assert_allclose(gate[:, 0], p[np.arange(T), am], rtol=1e-13)
    assert np.all(gate[:, 0] <= 1.0) and np.any(gate[:, 0] < 1.0)  # not renormalised


def pin_mask_renormalise(orc):
    """Softmax(KeepTopK(H)) equals the dense softmax masked to the top k and
    renormalised (the paper's appendix form, quoted in the lesson's Ch. 2)."""
    rng = np.random.default_rng(4)
    H = rng.standard_normal((40, 9)) * 2.0
    for k in (1, 2, 4, 9):
        idx, gate, _, _ = orc.select(H, k, TOPK)
        Gs = np.exp(H - H.max(axis=1, keepdims=True))
        Gs /= Gs.sum(axis=1, keepdims=True)
        M = np.zeros_like(H)
        np.put_along_axis(M, idx.astype(np.int64), 1.0, axis=1)
        ref = Gs * M / (Gs * M).sum(axis=1, keepdims=True)
        np.testing.assert_allclose(_dense_gates(idx, gate, 9), ref, rtol=1e-12, atol=1e-15)


def pin_gates_given(orc):
    rng = np.random.default_rng(5)
    H = rng.standard_normal((20, 7))
    for k, mode in ((1, SWITCH), (3, TOPK)):
        idx, gate, _, _ = orc.select(H, k, mode)
        np.testing.assert_allclose(orc.gates_given(H, idx, mode), gate, rtol=1e-14)


# ----------------------------------------------------------------------------- capacity, slots


def pin_capacity(orc):
    cases = [  # (T, E, k, cf, expected): the five measured workloads, then the clamps
        (8, 3, 1, 1.0, 2), (4096, 16, 4, 2.0, 2048), (16384, 64, 1, 1.25, 320),
        (8192, 8, 2, 1.25, 2560), (32768, 1024, 4, 1.5, 192),
        (2, 8, 1, 1.0, 1),  # floor(0.25) = 0 -> minimum 1
        (4, 1, 1, 2.0, 4),  # floor(8) -> clamped to T
    ]
    for T, E, k, cf, want in cases:
        exact = math.floor(Fraction(k * T) * Fraction(cf) / E)
        assert max(1, min(T, exact)) == want
        assert orc.capacity(T, E, k, cf, 1) == want, (T, E, k, cf)


def pin_slots_cumsum(orc):
    """Positions equal the exclusive cumulative sum of one-hot choices in
    token order (Switch step 3), accept iff position < C (step 4)."""
    rng = np.random.default_rng(6)
    T, k, E = 40, 3, 5
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[:10, 0] = 2  # pile onto one expert so that small capacities drop
    for C in (1, 3, 7, 1000):
        pos, keep, count = orc.slots(idx, E, C)
        onehot = np.zeros((T * k, E), np.int64)
        onehot[np.arange(T * k), idx.reshape(-1)] = 1
        excl = np.cumsum(onehot, axis=0) - onehot
        pos_ref = (excl * onehot).sum(axis=1).reshape(T, k)
        assert np.array_equal(pos, pos_ref)
        assert np.array_equal(keep.astype(bool), pos_ref < C)
        assert np.array_equal(count, onehot.sum(axis=0))
        assert int(keep.sum()) == int(np.minimum(onehot.sum(axis=0), C).sum())
        taken = {(int(idx[t, j]), int(pos[t, j])) for t in range(T) for j in range(k) if keep[t, j]}
        assert len(taken) == int(keep.sum())  # each slot holds at most one assignment


# ----------------------------------------------------------------------------- expert FFN and combine


def _small_case(rng, T, d, E, d_ff, bf16, biases=True):
    x = rng.standard_normal((T, d)).astype(np.float32)
    W1 = (rng.standard_normal((E, d, d_ff)) / math.sqrt(d)).astype(np.float32)
    W2 = (rng.standard_normal((E, d_ff, d)) / math.sqrt(d_ff)).astype(np.float32)
    b1 = (0.1 * rng.standard_normal((E, d_ff))).astype(np.float32) if biases else None
    b2 = (0.1 * rng.standard_normal((E, d))).astype(np.float32) if biases else None
    if bf16:
        x, W1, W2 = (f32_to_bf16_bits(a) for a in (x, W1, W2))
        b1 = None if b1 is None else f32_to_bf16_bits(b1)
        b2 = None if b2 is None else f32_to_bf16_bits(b2)
    return x, W1, b1, W2, b2


def pin_dense_sum(orc):
    """With nothing dropped, the per-token loop over kept experts equals the
    dense all-experts sum x + sum_e G_e E_e(x) (the MoE output equation), with
    G = Softmax(KeepTopK(H)) built independently in numpy."""
    rng = np.random.default_rng(7)
    T, d, E, d_ff, k = 6, 5, 4, 7, 2
    for bf16 in (False, True):
        x, W1, b1, W2, b2 = _small_case(rng, T, d, E, d_ff, bf16)
        H = rng.standard_normal((T, E))
        idx, gate, _, _ = orc.select(H, k, TOPK)
        keep = np.ones((T, k), np.uint8)
        y, bad = orc.layer_out(x, idx, gate, keep, W1, W2, b1, b2)
        assert not bad
        masked = np.full_like(H, -np.inf)
        for t in range(T):
            top = _ref_order(list(H[t]), k)
            masked[t, top] = H[t, top]
        G = np.exp(masked - masked.max(axis=1, keepdims=True))
        G /= G.sum(axis=1, keepdims=True)
        X = _x64(x)
        Y = _ffn_all(X, W1, b1, W2, b2)
        ref = X + np.einsum("te,etd->td", G, Y)
        np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12)


def pin_switch_einsum_algebra(orc):
    """With drops, the output equals the Switch page's dispatch / combine
    tensor algebra (steps 5-7) evaluated with numpy einsum."""
    rng = np.random.default_rng(8)
    T, d, E, d_ff = 10, 4, 3, 6
    for k in (1, 2):
        x, W1, b1, W2, b2 = _small_case(rng, T, d, E, d_ff, False)
        H = rng.standard_normal((T, E))
        H[:, 1] += 1.5  # overload expert 1
        mode = SWITCH if k == 1 else TOPK
        idx, gate, _, _ = orc.select(H, k, mode)
        C = 3
        onehot = np.zeros((T * k, E), np.int64)
        onehot[np.arange(T * k), idx.reshape(-1)] = 1
        pos = ((np.cumsum(onehot, axis=0) - onehot) * onehot).sum(axis=1).reshape(T, k)
        keep = (pos < C).astype(np.uint8)
        assert keep.sum() < T * k  # something overflowed
        dispatch = np.zeros((T, E, C))
        combine = np.zeros((T, E, C))
        for t in range(T):
            for j in range(k):
                if keep[t, j]:
                    dispatch[t, idx[t, j], pos[t, j]] = 1.0
                    combine[t, idx[t, j], pos[t, j]] = gate[t, j]
        X = _x64(x)
        U = np.einsum("tec,td->ecd", dispatch, X)
        Hh = np.maximum(np.einsum("ecd,edh->ech", U, W1.astype(np.float64)) + b1[:, None, :], 0.0)
        Z = np.einsum("ech,ehd->ecd", Hh, W2.astype(np.float64)) + b2[:, None, :]
        ref = X + np.einsum("tec,ecd->td", combine, Z)
        y, _ = orc.layer_out(x, idx, gate, keep, W1, W2, b1, b2)
        np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12)


def pin_dropped_identity(orc):
    """A token whose choices all overflow leaves the layer unchanged."""
    rng = np.random.default_rng(9)
    T, d, E, d_ff = 8, 6, 3, 5
    x, W1, b1, W2, b2 = _small_case(rng, T, d, E, d_ff, True)
    H = np.tile([3.0, 0.0, -1.0], (T, 1))
    idx, gate, _, _ = orc.select(H, 1, SWITCH)
    pos, keep, _ = orc.slots(idx, E, 2)
    y, _ = orc.layer_out(x, idx, gate, keep, W1, W2, b1, b2)
    X = _x64(x)
    assert np.array_equal(y[2:], X[2:])
    assert not np.array_equal(y[:2], X[:2])


def pin_dense_mlp_special_case(orc):
    """One expert, top-1 Switch, capacity T: every gate is Softmax over one
    expert = 1 and the layer is x + a plain two-layer ReLU MLP."""
    rng = np.random.default_rng(10)
    T, d, d_ff = 9, 6, 11
    x, W1, b1, W2, b2 = _small_case(rng, T, d, 1, d_ff, False)
    Wg = rng.standard_normal((d, 1)).astype(np.float32)
    c, s, H, _ = orc.router(x, Wg)
    idx, gate, _, _ = orc.select(H, 1, SWITCH)
    assert np.all(gate == 1.0)
    C = orc.capacity(T, 1, 1, 1.0, 1)
    assert C == T
    pos, keep, _ = orc.slots(idx, 1, C)
    y, _ = orc.layer_out(x, idx, gate, keep, W1, W2, b1, b2)
    X = _x64(x)
    ref = X + np.maximum(X @ W1[0].astype(np.float64) + b1[0], 0.0) @ W2[0].astype(np.float64) + b2[0]
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------------------------- balancing losses


def pin_cv(orc):
    for ex in GOLDEN["cv"]:
        assert abs(orc.cv2(ex["importance"]) - ex["cv2"]) <= ex["tol"], ex["source"]
    v = np.array([3.0, 1.0, 4.0, 1.0, 5.0])
    assert abs(orc.cv2(v) - np.var(v) / np.mean(v) ** 2) < 1e-14


def pin_importance_and_noise_free_load(orc):
    rng = np.random.default_rng(11)
    T, E, k = 30, 5, 2
    H = rng.standard_normal((T, E))
    idx, gate, hk, hk1 = orc.select(H, k, TOPK)
    zero = np.zeros_like(H)
    a = orc.aux(H, zero, H, idx, gate, hk, hk1, False)
    G = _dense_gates(idx, gate, E)
    np.testing.assert_allclose(a["importance"], G.sum(axis=0), rtol=1e-13)
    counts = np.bincount(idx.reshape(-1), minlength=E)
    assert np.array_equal(a["load"], counts.astype(np.float64))
    np.testing.assert_allclose(a["out3"][0], np.var(a["importance"]) / np.mean(a["importance"]) ** 2,
                               rtol=1e-12)
    np.testing.assert_allclose(a["out3"][1], np.var(counts) / np.mean(counts) ** 2, rtol=1e-12)
    idx, gate, hk, hk1 = orc.select(H, E, TOPK)  # k = E: every expert always chosen
    a = orc.aux(H, zero + 1.0, H, idx, gate, hk, hk1, True)
    assert np.all(a["load"] == T) and a["out3"][1] == 0.0


def pin_load_lesson_reading(orc):
    """The lesson's Ch. 5 load example: H = [2.3, 0.8, 0.6, -2.0], clean
    [2.0, 1.0, 0.5, -0.5], noise scale 1, k = 2. kth_excluding drops the expert
    and takes the 2nd largest of the rest ([0.6, 0.6, 0.8, 0.8]); P = Phi(clean -
    kth_excluding), evaluated here with scipy's normal CDF."""
    Hr = np.array([[2.3, 0.8, 0.6, -2.0]])
    clean = np.array([[2.0, 1.0, 0.5, -0.5]])
    idx, gate, hk, hk1 = orc.select(Hr, 2, TOPK)
    a = orc.aux(clean, np.ones_like(Hr), Hr, idx, gate, hk, hk1, True)
    kth = np.array([0.6, 0.6, 0.8, 0.8])
    np.testing.assert_allclose(a["load"], ndtr(clean[0] - kth), rtol=1e-13)


def pin_load_monte_carlo(orc):
    """P(x,i) is the probability that expert i stays in the top k when only
    its own noise is redrawn: count it by brute force."""
    rng = np.random.default_rng(12)
    T, E, k, N = 3, 5, 2, 40000
    c = rng.standard_normal((T, E))
    s = 0.3 + rng.random((T, E))
    n = rng.standard_normal((T, E))
    H = c + n * s
    idx, gate, hk, hk1 = orc.select(H, k, TOPK)
    a = orc.aux(c, s, H, idx, gate, hk, hk1, True)
    est = np.zeros(E)
    for t in range(T):
        for e in range(E):
            draws = c[t, e] + rng.standard_normal(N) * s[t, e]
            others = np.delete(H[t], e)
            beaten_by = (others[None, :] > draws[:, None]).sum(axis=1)
            est[e] += np.mean(beaten_by < k)
    tol = 5.0 * math.sqrt(T * 0.25 / N)
    assert np.all(np.abs(a["load"] - est) < tol), (a["load"], est)


def pin_switch_aux_closed_forms(orc):
    alpha = GOLDEN["switch_aux"]["alpha"]
    E, m = 4, 3
    v = np.array([1.0, 0.2, -0.3, 0.7])
    H = np.stack([np.roll(v, r) for r in range(E)] * m)  # every expert first equally often
    idx, gate, hk, hk1 = orc.select(H, 1, SWITCH)
    a = orc.aux(H, np.zeros_like(H), H, idx, gate, hk, hk1, False)
    np.testing.assert_allclose(a["f"], 1.0 / E, rtol=1e-14)
    np.testing.assert_allclose(a["pbar"], 1.0 / E, rtol=1e-13)
    assert abs(a["out3"][2] - alpha) < 1e-14
    H = np.tile(v, (7, 1))  # collapse: every token picks expert 0 with probability q
    idx, gate, hk, hk1 = orc.select(H, 1, SWITCH)
    a = orc.aux(H, np.zeros_like(H), H, idx, gate, hk, hk1, False)
    q = np.exp(v[0]) / np.exp(v).sum()
    assert abs(a["out3"][2] - alpha * E * q) < 1e-14


# ----------------------------------------------------------------------------- scalars, errors


def pin_softplus_phi(orc):
    for z in np.linspace(-50.0, 50.0, 41):
        assert abs(orc.softplus(z) - np.logaddexp(0.0, z)) <= 1e-14 * max(1.0, abs(z))
    assert orc.softplus(-10.0) > 0.0
    for u in np.linspace(-8.0, 8.0, 33):
        assert abs(orc.phi(u) - ndtr(u)) < 1e-15
    assert orc.phi(0.0) == 0.5


def pin_nonfinite(orc):
    x = np.ones((2, 3), np.float32)
    x[1, 2] = np.inf
    _, _, _, bad = orc.router(x, np.ones((3, 2), np.float32))
    assert bad
    W1 = np.ones((1, 3, 2), np.float32)
    W1[0, 0, 0] = np.nan
    y, bad = orc.layer_out(np.ones((1, 3), np.float32), np.zeros((1, 1), np.int32), np.ones((1, 1)),
                           np.ones((1, 1), np.uint8), W1, np.ones((1, 2, 3), np.float32))
    assert bad


# ----------------------------------------------------------------------------- hierarchical


def _hier_case(rng, T, d, a, b, d_ff, noisy=True):
    x = rng.standard_normal((T, d)).astype(np.float32)
    sd = 1.0 / math.sqrt(d)
    E = a * b
    inp = dict(x=x, Wp=(rng.standard_normal((d, a)) * sd).astype(np.float32),
               Ws=(rng.standard_normal((d, E)) * sd).astype(np.float32),
               Wpn=None, noise_p=None, Wsn=None, noise_s=None)
    if noisy:
        inp.update(Wpn=(rng.standard_normal((d, a)) * sd).astype(np.float32),
                   noise_p=rng.standard_normal((T, a)).astype(np.float32),
                   Wsn=(rng.standard_normal((d, E)) * sd).astype(np.float32),
                   noise_s=rng.standard_normal((T, E)).astype(np.float32))
    _, W1, b1, W2, b2 = _small_case(rng, T, d, E, d_ff, False)
    inp.update(W1=W1, b1=b1, W2=W2, b2=b2, a=a, b=b, cf=float(E), min_cap=1)
    return inp


def _np_logits(X, W, Wn, noise):
    """c, sigma, H of a noisy gate in numpy (OLNN Eq. 4)."""
    c = X @ W.astype(np.float64)
    if Wn is None:
        return c, np.zeros_like(c), c
    s = np.logaddexp(0.0, X @ Wn.astype(np.float64))
    return c, s, c + noise.astype(np.float64) * s


def _np_topk_gate(h, k):
    """Dense Softmax(KeepTopK(h, k)) and the ordered picks."""
    top = _ref_order(list(h), k)
    g = np.zeros(len(h))
    ex = np.exp(h[top] - h[top[0]])
    g[top] = ex / ex.sum()
    return g, top


def _np_smooth_load(c, s, h, k, members=None):
    """sum over rows of P(x, e) = Phi((c_e - kth_excluding(h, k, e)) / s_e)
    (OLNN Eqs. 8-9), computed row by row in numpy/scipy; rows limited to
    ``members`` when given."""
    T, E = h.shape
    out = np.zeros(E)
    for t in range(T) if members is None else members:
        for e in range(E):
            others = np.sort(np.delete(h[t], e))[::-1]
            if k >= E:
                out[e] += 1.0
            elif s[t, e] == 0.0:
                out[e] += 1.0 if e in _ref_order(list(h[t]), k) else 0.0
            else:
                out[e] += ndtr((c[t, e] - others[k - 1]) / s[t, e])
    return out


def pin_hier_dense_formula(orc):
    """The hierarchical layer against its definition written out densely in
    numpy on a tiny case (OLNN "Hierarchical Mixture-of-Experts"):
    y_H = x + sum_i sum_j G_p(x)_i G_i(x)_j E_ij(x), Importance_H = sum of the
    products, Load_H = Load_p(X)_i Load_i(X^(i))_j / |X^(i)|, with every gate
    a noisy top-k softmax and every load the smooth estimator, and nothing
    dropped (capacity T)."""
    rng = np.random.default_rng(41)
    T, d, a, b, kp, ks, d_ff = 9, 6, 3, 4, 2, 2, 5
    inp = _hier_case(rng, T, d, a, b, d_ff)
    inp.update(kp=kp, ks=ks)
    r = orc.hier_forward(inp)
    X = _x64(inp["x"])
    cp, sp, Hp = _np_logits(X, inp["Wp"], inp["Wpn"], inp["noise_p"])
    cs, ss, Hs = _np_logits(X, inp["Ws"], inp["Wsn"], inp["noise_s"])
    Y = _ffn_all(X, inp["W1"], inp["b1"], inp["W2"], inp["b2"])
    y_ref = X.copy()
    imp = np.zeros(a * b)
    members = [[] for _ in range(a)]
    for t in range(T):
        gp, picks = _np_topk_gate(Hp[t], kp)
        for i in picks:
            members[i].append(t)
            gi, _ = _np_topk_gate(Hs[t, i * b:(i + 1) * b], ks)
            for j in range(b):
                w = gp[i] * gi[j]
                y_ref[t] += w * Y[i * b + j, t]
                imp[i * b + j] += w
    np.testing.assert_allclose(r["y"], y_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(r["importance_H"], imp, rtol=1e-12, atol=1e-14)
    load_p = _np_smooth_load(cp, sp, Hp, kp)
    load_H = np.zeros(a * b)
    for i in range(a):
        sec = _np_smooth_load(cs[:, i * b:(i + 1) * b], ss[:, i * b:(i + 1) * b],
                              Hs[:, i * b:(i + 1) * b], ks, members[i])
        if members[i]:
            load_H[i * b:(i + 1) * b] = load_p[i] * sec / len(members[i])
    assert list(r["group_count"]) == [len(m) for m in members]
    np.testing.assert_allclose(r["load_H"], load_H, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(r["out2"], [np.var(imp) / np.mean(imp) ** 2,
                                           np.var(load_H) / np.mean(load_H) ** 2], rtol=1e-10)


def pin_hier_one_group_is_flat(orc):
    """a = 1, kp = 1: the primary gate is 1 for every token, so the layer,
    Importance_H and Load_H are the flat layer's over the b experts."""
    rng = np.random.default_rng(43)
    T, d, b, ks, d_ff = 20, 7, 6, 2, 4
    inp = _hier_case(rng, T, d, 1, b, d_ff)
    inp.update(kp=1, ks=ks, cf=1.0)
    r = orc.hier_forward(inp)
    flat = orc.forward(dict(x=inp["x"], Wg=inp["Ws"], Wn=inp["Wsn"], noise=inp["noise_s"],
                            bias=None, W1=inp["W1"], b1=inp["b1"], W2=inp["W2"], b2=inp["b2"],
                            k=ks, cf=1.0, min_cap=1, mode=TOPK))
    assert np.array_equal(r["idx"], flat["idx"]) and np.array_equal(r["keep"], flat["keep"])
    np.testing.assert_allclose(r["gate"], flat["gate"], rtol=1e-14)
    np.testing.assert_allclose(r["y"], flat["y"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(r["importance_H"], flat["importance"], rtol=1e-13)
    np.testing.assert_allclose(r["load_H"], flat["load"], rtol=1e-12)
    np.testing.assert_allclose(r["out2"], flat["out3"][:2], rtol=1e-10)


def pin_hier_single_expert_groups(orc):
    """b = 1, ks = 1: every secondary gate is 1, so the layer is the flat
    layer over the a groups; Importance_H is the primary importance and
    Load_H the primary load wherever the group was picked."""
    rng = np.random.default_rng(47)
    T, d, a, kp, d_ff = 40, 5, 4, 2, 3
    inp = _hier_case(rng, T, d, a, 1, d_ff)
    inp.update(kp=kp, ks=1, cf=2.0)
    r = orc.hier_forward(inp)
    flat = orc.forward(dict(x=inp["x"], Wg=inp["Wp"], Wn=inp["Wpn"], noise=inp["noise_p"],
                            bias=None, W1=inp["W1"], b1=inp["b1"], W2=inp["W2"], b2=inp["b2"],
                            k=kp, cf=2.0, min_cap=1, mode=TOPK))
    assert np.array_equal(r["idx"], flat["idx"])
    np.testing.assert_allclose(r["y"], flat["y"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(r["importance_H"], flat["importance"], rtol=1e-13)
    assert np.all(r["group_count"] > 0)
    np.testing.assert_allclose(r["load_H"], flat["load"], rtol=1e-12)


def pin_hier_empty_group_guard(orc):
    """A group that no token's primary gate picks has |X^(i)| = 0, and its
    Load_H entries are 0 (the quotient is undefined there); the product gates
    of every token sum to 1, so Importance_H sums to T."""
    rng = np.random.default_rng(53)
    T, d, a, b, kp, ks, d_ff = 25, 3, 3, 4, 2, 2, 3
    inp = _hier_case(rng, T, d, a, b, d_ff, noisy=False)
    x = inp["x"].copy()
    x[:, 0] = 1.0
    inp["x"] = x
    Wp = np.zeros((d, a), np.float32)
    Wp[0] = [5.0, 4.0, -10.0]  # group 2 is always the lowest of the three
    inp.update(Wp=Wp, kp=kp, ks=ks)
    r = orc.hier_forward(inp)
    assert list(r["group_count"]) == [T, T, 0]
    assert np.all(r["load_H"][2 * b:] == 0.0)
    assert np.all(np.isfinite(r["load_H"]))
    np.testing.assert_allclose(r["importance_H"].sum(), T, rtol=1e-13)
    # noise-free: Load_H of a picked group is the in-group pick count (the
    # primary load of a group picked by every token is T = |X^(i)|)
    cnt = np.bincount(r["idx"].reshape(-1), minlength=a * b).astype(np.float64)
    np.testing.assert_allclose(r["load_H"][:2 * b], cnt[:2 * b], rtol=1e-13)


# ----------------------------------------------------------------------------- strictly balanced


def pin_softmax_rows(orc):
    """The plain softmax gate against scipy's softmax, including logits large
    enough to overflow exp without the max shift."""
    from scipy.special import softmax
    rng = np.random.default_rng(71)
    H = rng.standard_normal((6, 9)) * 3.0
    H[2] += 900.0
    np.testing.assert_allclose(orc.softmax_dense(H), softmax(H, axis=1), rtol=1e-13, atol=1e-300)


def _bal_ref_mask(P, m):
    T, E = P.shape
    M = np.zeros((T, E), np.uint8)
    for i in range(E):
        for t in sorted(range(T), key=lambda u: (-P[u, i], u))[:m]:
            M[t, i] = 1
    return M


def pin_bal_rows_lesson(orc):
    """The lesson's translation-scale pooling example (golden fixture): k = 2,
    n = 512 experts, 16,000 words on one GPU give 62.5 per expert (a mask
    takes whole tokens: 62), and pooled over 64 GPUs exactly 4,000; plus the
    clamps to 1 and to T."""
    for ex in GOLDEN["batchwise_rows"]:
        m = orc.bal_rows(ex["T"], ex["k"], ex["E"])
        assert m == math.floor(ex["per_expert"]), (ex["source"], m)
    assert orc.bal_rows(3, 1, 8) == 1 and orc.bal_rows(5, 8, 4) == 5


def pin_bal_batchwise_bruteforce(orc):
    """The batchwise mask: per expert the m tokens with the largest dense gate
    (Python sort by (-P, token), ties included); every expert exactly m; gates
    P * M renormalised per token, 0 for a token no expert took."""
    rng = np.random.default_rng(73)
    T, E, m = 11, 5, 4
    P = rng.random((T, E))
    P /= P.sum(axis=1, keepdims=True)
    top = -np.sort(-P[:, 1])
    P[3, 1] = P[7, 1] = P[9, 1] = top[2]  # a three-way tie across the m-th place
    P[0, 2] = P[10, 2] = -np.sort(-P[:, 2])[m - 1]
    mask, gate = orc.bal_gate(P, m)
    ref = _bal_ref_mask(P, m)
    assert np.array_equal(mask, ref)
    assert np.all(mask.sum(axis=0) == m)
    z = (P * ref).sum(axis=1, keepdims=True)
    g_ref = np.where(ref == 1, P / np.where(z > 0, z, 1.0), 0.0)
    np.testing.assert_allclose(gate, g_ref, rtol=1e-14, atol=0)
    assert np.all(gate[ref.sum(axis=1) == 0] == 0.0)


def pin_bal_threshold_mask_and_loss(orc):
    """The threshold mask P > T_i and L_batchwise: with each T_i between the
    m-th and (m+1)-th largest P of its column both masks agree and the loss
    is exactly 0; lowering one threshold past one more token adds exactly
    P - T_i for that token; P equal to its threshold is not taken."""
    rng = np.random.default_rng(79)
    T, E, m = 12, 4, 3
    H = rng.standard_normal((T, E))
    P = orc.softmax_dense(H)
    mb, _ = orc.bal_gate(P, m)
    srt = -np.sort(-P, axis=0)
    thr = ((srt[m - 1] + srt[m]) / 2).astype(np.float32)
    mt, _ = orc.bal_gate(P, m, thr, 1)
    assert np.array_equal(mt, (P > thr.astype(np.float64)[None, :]).astype(np.uint8))
    assert np.array_equal(mt, mb)
    assert orc.bal_loss(P, mb, thr) == 0.0
    thr2 = thr.copy()
    thr2[1] = np.float32((srt[m, 1] + srt[m + 1, 1]) / 2)
    extra = np.nonzero((P[:, 1] > thr2[1]) & (mb[:, 1] == 0))[0]
    assert extra.size == 1
    want = sum((float(P[t, i] > thr2[i]) - mb[t, i]) * (P[t, i] - float(thr2[i]))
               for t in range(T) for i in range(E))
    np.testing.assert_allclose(orc.bal_loss(P, mb, thr2), want, rtol=1e-13)
    assert orc.bal_loss(P, mb, thr2) > 0.0
    half = orc.softmax_dense(np.zeros((1, 2)))  # exactly 0.5 each
    mh, _ = orc.bal_gate(half, 1, np.array([0.5, 0.25], np.float32), 1)
    assert list(mh[0]) == [0, 1]


def pin_bal_every_token_is_dense(orc):
    """m = T (k = E): every expert takes every token, the gate is the dense
    softmax itself, and the layer is the dense soft mixture x + sum_i
    G_sigma(x)_i E_i(x) (numpy)."""
    rng = np.random.default_rng(83)
    T, d, E, d_ff = 7, 5, 3, 4
    x, W1, b1, W2, b2 = _small_case(rng, T, d, E, d_ff, False)
    Wg = (rng.standard_normal((d, E)) / math.sqrt(d)).astype(np.float32)
    r = orc.bal_forward(dict(x=x, Wg=Wg, W1=W1, b1=b1, W2=W2, b2=b2, k=E))
    assert r["m"] == T and np.all(r["mask"] == 1)
    X = _x64(x)
    H = X @ Wg.astype(np.float64)
    G = np.exp(H - H.max(axis=1, keepdims=True))
    G /= G.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(r["gate"], G, rtol=1e-13)
    ref = X + np.einsum("te,etd->td", G, _ffn_all(X, W1, b1, W2, b2))
    np.testing.assert_allclose(r["y"], ref, rtol=1e-11, atol=1e-12)



# ----------------------------------------------------------------------------- backward


def _grad_case(seed, T, d, E, d_ff, k, cf, mode, noisy, router_bias=True, biases=True):
    """fp32 inputs for the gradient pins: every weight is an fp32 value, so a
    step of 2^-12 on any entry below 2^11 in magnitude is exact."""
    rng = np.random.default_rng(seed)
    f = lambda *sh, sd=1.0: (rng.standard_normal(sh) * sd).astype(np.float32)
    inp = dict(x=f(T, d), Wg=f(d, E, sd=1 / math.sqrt(d)), k=k, cf=cf, min_cap=1, mode=mode,
               W1=f(E, d, d_ff, sd=1 / math.sqrt(d)), W2=f(E, d_ff, d, sd=1 / math.sqrt(d_ff)))
    inp["Wn"] = f(d, E, sd=1 / math.sqrt(d)) if noisy else None
    inp["noise"] = f(T, E) if noisy else None
    inp["bias"] = f(E, sd=0.3) if router_bias else None
    inp["b1"] = f(E, d_ff, sd=0.1) if biases else None
    inp["b2"] = f(E, d, sd=0.1) if biases else None
    dy = rng.standard_normal((T, d))
    return inp, dy


_GRAD_OF = dict(x="dx", Wg="dWg", Wn="dWn", bias="dbias", W1="dW1", b1="db1", W2="dW2", b2="db2")


def _finite_difference_check(orc, inp, dy, w, per_param, seed):
    """Central differences of the forward's scalar loss on sampled entries of
    every input. The forward's discrete choices (top-k, capacity, ReLU) make
    the loss piecewise smooth; an entry whose one-sided differences disagree
    sits on a kink (or has a gradient near zero, where curvature alone
    separates them) and is skipped: at most 3, or one in eight."""
    g = orc.backward(inp, dy, *w)
    L0 = orc.loss(inp, dy, *w)
    eps = 2.0 ** -12
    rng = np.random.default_rng(seed)
    checked = skipped = 0
    for name, gname in _GRAD_OF.items():
        a = inp.get(name)
        if a is None:
            continue
        for _ in range(per_param):
            i = tuple(int(rng.integers(0, n)) for n in a.shape)
            v = a[i]
            a[i] = v + np.float32(eps)
            Lp = orc.loss(inp, dy, *w)
            a[i] = v - np.float32(eps)
            Lm = orc.loss(inp, dy, *w)
            a[i] = v
            up, down = (Lp - L0) / eps, (L0 - Lm) / eps
            if abs(up - down) > 1e-3 * (abs(up) + abs(down)) + 1e-6:
                skipped += 1
                continue
            fd = (Lp - Lm) / (2 * eps)
            assert abs(g[gname][i] - fd) <= 1e-5 * abs(fd) + 1e-7, (name, i, g[gname][i], fd)
            checked += 1
    assert skipped <= max(3, checked // 8), (checked, skipped)


def pin_backward_finite_differences(orc):
    """The backward equals central differences of the forward's loss, for
    noisy top-k with capacity drops and all three balancing terms, clean and
    noisy Switch top-1 with the auxiliary loss, and k = E (no load gradient)."""
    cases = [
        (_grad_case(101, 12, 6, 5, 7, 2, 0.8, TOPK, True), (0.7, 0.9, 0.4)),
        (_grad_case(102, 10, 5, 4, 6, 1, 0.9, SWITCH, False), (0.3, 0.2, 0.8)),
        (_grad_case(103, 10, 5, 4, 6, 1, 0.9, SWITCH, True), (0.3, 0.6, 0.8)),
        (_grad_case(104, 9, 5, 6, 4, 3, 2.0, TOPK, True, router_bias=False, biases=False),
         (1.0, 1.0, 1.0)),
        (_grad_case(105, 8, 4, 3, 5, 3, 2.0, TOPK, True), (1.0, 1.0, 1.0)),
    ]
    for n, ((inp, dy), w) in enumerate(cases):
        fw = orc.forward(inp)
        if n == 0:  # the case must exercise capacity drops
            assert fw["keep"].min() == 0 and fw["keep"].max() == 1
        _finite_difference_check(orc, inp, dy, w, 12, 200 + n)


def pin_backward_dense_mlp(orc):
    """One expert: every gate is 1, the balancing terms are constant, and the
    gradients are those of x + ReLU(x W1 + b1) W2 + b2 in matrix form (numpy);
    the router weights get none."""
    for mode in (TOPK, SWITCH):
        inp, dy = _grad_case(110 + mode, 9, 6, 1, 11, 1, 1.0, mode, True)
        g = orc.backward(inp, dy, 0.5, 0.5, 0.5)
        X = inp["x"].astype(np.float64)
        W1, W2 = inp["W1"][0].astype(np.float64), inp["W2"][0].astype(np.float64)
        pre = X @ W1 + inp["b1"][0]
        h = np.maximum(pre, 0.0)
        dpre = (dy @ W2.T) * (pre > 0)
        np.testing.assert_allclose(g["dW2"][0], h.T @ dy, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(g["db2"][0], dy.sum(0), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(g["dW1"][0], X.T @ dpre, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(g["db1"][0], dpre.sum(0), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(g["dx"], dy + dpre @ W1.T, rtol=1e-12, atol=1e-12)
        for name in ("dWg", "dWn", "dbias"):
            assert np.all(g[name] == 0.0), name


def pin_backward_logit_shift_invariance(orc):
    """Adding one constant to every expert's router logit of a token changes
    neither the gates, the selection, the load estimator's arguments c - thr
    nor the full softmax, so the gradient summed over experts vanishes: for
    the router bias and for every row of W_g."""
    for seed, (T, d, E, d_ff, k, cf, mode, noisy) in enumerate(
            [(12, 6, 5, 7, 2, 0.8, TOPK, True), (10, 5, 4, 6, 1, 0.9, SWITCH, True)]):
        inp, dy = _grad_case(120 + seed, T, d, E, d_ff, k, cf, mode, noisy)
        g = orc.backward(inp, dy, 0.7, 0.9, 0.4)
        scale = np.abs(g["dbias"]).sum()
        assert scale > 1e-3
        assert abs(g["dbias"].sum()) <= 1e-12 * scale + 1e-15
        rows = g["dWg"].sum(axis=1)
        assert np.all(np.abs(rows) <= 1e-12 * np.abs(g["dWg"]).sum(axis=1) + 1e-15)



def pin_backward_dgate(orc):
    """dL/dgate of a selected choice: <dy_t, E_e(x_t)> (numpy expert) when it
    is kept, 0 when it overflowed, plus w_imp times the derivative of
    CV(Importance)^2 in that expert's importance (central differences of the
    pinned CV^2), which is the same for every choice of one expert."""
    inp, dy = _grad_case(130, 12, 6, 5, 7, 2, 0.8, TOPK, True)
    fw = orc.forward(inp)
    assert fw["keep"].min() == 0
    X = inp["x"].astype(np.float64)
    U = _ffn_all(X, inp["W1"], inp["b1"], inp["W2"], inp["b2"])  # [E, T, d]
    g0 = orc.backward(inp, dy, 0.0, 0.0, 0.0)["dgate"]
    for t in range(X.shape[0]):
        for j in range(2):
            e = fw["idx"][t, j]
            want = float(dy[t] @ U[e, t]) if fw["keep"][t, j] else 0.0
            assert abs(g0[t, j] - want) <= 1e-12 * (1 + abs(want)), (t, j)
    w = 0.7
    g1 = orc.backward(inp, dy, w, 0.0, 0.0)["dgate"]
    imp = fw["importance"]
    h = 1e-6
    for e in range(imp.size):
        up, dn = imp.copy(), imp.copy()
        up[e] += h
        dn[e] -= h
        want = w * (orc.cv2(up) - orc.cv2(dn)) / (2 * h)
        sel = fw["idx"] == e
        if sel.any():
            np.testing.assert_allclose((g1 - g0)[sel], want, rtol=1e-6, atol=1e-9)



def pin_backward_entries(orc):
    """The entry-by-entry weight gradients (sums over the expert's kept rows)
    equal orc_backward's on a layer with capacity drops, bf16 weights and
    biases; the sums of |terms| bound the entries."""
    inp, dy = _grad_case(140, 14, 6, 4, 10, 2, 0.8, TOPK, True)
    for n in ("x", "W1", "W2", "b1", "b2"):
        inp[n] = f32_to_bf16_bits(inp[n])
    ref = orc.backward(inp, dy, 0.3, 0.4, 0.5)
    rng = np.random.default_rng(141)
    entries = []
    for _ in range(12):
        e = int(rng.integers(4))
        entries += [("dW1", e, int(rng.integers(6)), int(rng.integers(10))),
                    ("dW2", e, int(rng.integers(10)), int(rng.integers(6))),
                    ("db1", e, int(rng.integers(10)), 0), ("db2", e, int(rng.integers(6)), 0)]
    got, absum = orc.backward_entries(inp, dy, entries)
    for (kind, e, a, b), v, m in zip(entries, got, absum):
        want = ref[kind][e, a, b] if kind in ("dW1", "dW2") else ref[kind][e, a]
        assert abs(v - want) <= 1e-12 * (1 + abs(want)), (kind, e, a, b, v, want)
        assert abs(v) <= m * (1 + 1e-12)



def _hier_grad_case(seed, T, d, a, b, kp, ks, d_ff, cf, noisy):
    rng = np.random.default_rng(seed)
    f = lambda *sh, sd=1.0: (rng.standard_normal(sh) * sd).astype(np.float32)
    E = a * b
    inp = dict(x=f(T, d), Wp=f(d, a, sd=1 / math.sqrt(d)), Ws=f(d, E, sd=1 / math.sqrt(d)),
               W1=f(E, d, d_ff, sd=1 / math.sqrt(d)), W2=f(E, d_ff, d, sd=1 / math.sqrt(d_ff)),
               b1=f(E, d_ff, sd=0.1), b2=f(E, d, sd=0.1), a=a, b=b, kp=kp, ks=ks, cf=cf,
               min_cap=1)
    inp["Wpn"] = f(d, a, sd=1 / math.sqrt(d)) if noisy else None
    inp["noise_p"] = f(T, a) if noisy else None
    inp["Wsn"] = f(d, E, sd=1 / math.sqrt(d)) if noisy else None
    inp["noise_s"] = f(T, E) if noisy else None
    return inp, rng.standard_normal((T, d))


def pin_hier_backward_finite_differences(orc):
    """The hierarchical backward equals central differences of the
    hierarchical forward's loss (noisy, with capacity drops; clean; one
    primary pick of two groups)."""
    names = dict(x="dx", Wp="dWp", Wpn="dWpn", Ws="dWs", Wsn="dWsn", W1="dW1", b1="db1",
                 W2="dW2", b2="db2")
    cases = [((150, 12, 5, 3, 4, 2, 2, 6, 0.7, True), (0.7, 0.9)),
             ((151, 10, 5, 3, 4, 2, 2, 6, 0.7, False), (0.5, 0.5)),
             ((152, 12, 5, 2, 5, 1, 3, 6, 0.9, True), (0.6, 0.8))]
    for n, (args, w) in enumerate(cases):
        inp, dy = _hier_grad_case(*args)
        g = orc.hier_backward(inp, dy, *w)
        L0 = orc.hier_loss(inp, dy, *w)
        eps = 2.0 ** -12
        rng = np.random.default_rng(160 + n)
        checked = skipped = 0
        for name, gname in names.items():
            A = inp.get(name)
            if A is None:
                continue
            for _ in range(10):
                i = tuple(int(rng.integers(0, m)) for m in A.shape)
                v = A[i]
                A[i] = v + np.float32(eps)
                Lp = orc.hier_loss(inp, dy, *w)
                A[i] = v - np.float32(eps)
                Lm = orc.hier_loss(inp, dy, *w)
                A[i] = v
                up, down = (Lp - L0) / eps, (L0 - Lm) / eps
                if abs(up - down) > 1e-3 * (abs(up) + abs(down)) + 1e-6:
                    skipped += 1
                    continue
                fd = (Lp - Lm) / (2 * eps)
                assert abs(g[gname][i] - fd) <= 1e-5 * abs(fd) + 1e-7, (n, name, i, g[gname][i], fd)
                checked += 1
        assert skipped <= max(2, checked // 10), (checked, skipped)


def pin_hier_backward_one_group_is_flat(orc):
    """One group (a = 1, kp = 1): the primary gate is the constant 1, Load_H
    is the flat load, and the hierarchical backward equals the flat layer's
    backward over the b experts; the primary router gets no gradient."""
    inp, dy = _hier_grad_case(170, 11, 5, 1, 5, 1, 2, 6, 0.8, True)
    g = orc.hier_backward(inp, dy, 0.6, 0.7)
    flat = dict(x=inp["x"], Wg=inp["Ws"], Wn=inp["Wsn"], noise=inp["noise_s"], bias=None,
                W1=inp["W1"], b1=inp["b1"], W2=inp["W2"], b2=inp["b2"], k=2, cf=0.8, min_cap=1,
                mode=TOPK)
    ref = orc.backward(flat, dy, 0.6, 0.7, 0.0)
    for hn, fn in (("dx", "dx"), ("dWs", "dWg"), ("dWsn", "dWn"), ("dW1", "dW1"), ("db1", "db1"),
                   ("dW2", "dW2"), ("db2", "db2")):
        np.testing.assert_allclose(g[hn], ref[fn], rtol=1e-10, atol=1e-12, err_msg=hn)
    assert np.all(np.abs(g["dWp"]) <= 1e-12) and np.all(np.abs(g["dWpn"]) <= 1e-12)



def pin_bal_backward_finite_differences(orc):
    """The strictly balanced layer's backward equals central differences of
    its forward's loss sum <dy, y> + w L_batchwise: batchwise mask with the
    loss, the threshold mask as the gate, and every expert taking every token
    (k = E)."""
    names = dict(x="dx", Wg="dWg", bias="dbias", W1="dW1", b1="db1", W2="dW2", b2="db2")
    for n, (T, E, k, mode, w) in enumerate([(12, 4, 2, 0, 0.7), (12, 4, 2, 1, 0.5),
                                            (9, 3, 3, 0, 0.3)]):
        rng = np.random.default_rng(180 + n)
        f = lambda *sh, sd=1.0: (rng.standard_normal(sh) * sd).astype(np.float32)
        d, d_ff = 5, 6
        inp = dict(x=f(T, d), Wg=f(d, E, sd=1.5 / math.sqrt(d)), bias=f(E, sd=0.3),
                   W1=f(E, d, d_ff, sd=1 / math.sqrt(d)), W2=f(E, d_ff, d, sd=1 / math.sqrt(d_ff)),
                   b1=f(E, d_ff, sd=0.1), b2=f(E, d, sd=0.1), k=k, mode_bal=mode,
                   thr=np.full(E, 1.0 / E, np.float32))
        dy = rng.standard_normal((T, d))
        g = orc.bal_backward(inp, dy, w)
        L0 = orc.bal_loss_total(inp, dy, w)
        eps = 2.0 ** -12
        checked = skipped = 0
        for name, gname in names.items():
            A = inp[name]
            for _ in range(10):
                i = tuple(int(rng.integers(0, m)) for m in A.shape)
                v = A[i]
                A[i] = v + np.float32(eps)
                Lp = orc.bal_loss_total(inp, dy, w)
                A[i] = v - np.float32(eps)
                Lm = orc.bal_loss_total(inp, dy, w)
                A[i] = v
                up, down = (Lp - L0) / eps, (L0 - Lm) / eps
                if abs(up - down) > 1e-3 * (abs(up) + abs(down)) + 1e-6:
                    skipped += 1
                    continue
                fd = (Lp - Lm) / (2 * eps)
                assert abs(g[gname][i] - fd) <= 1e-5 * abs(fd) + 1e-7, (n, name, i, g[gname][i], fd)
                checked += 1
        assert skipped <= max(2, checked // 10), (checked, skipped)



def pin_backward_varied_layers(orc):
    """Central differences of the backward on more small layers: one expert,
    k = E with noise, top-2 of 5 with heavy drops (cf = 0.5) and biases,
    top-4 of 6 without noise but with a router bias, noisy Switch with drops,
    and noisy top-1 of 2."""
    layers = [  # (E, mode, k, T, d, d_ff, cf, noisy, router_bias, biases)
        (1, TOPK, 1, 7, 4, 5, 1.0, True, False, True),
        (3, TOPK, 3, 8, 4, 5, 1.0, True, True, False),
        (5, TOPK, 2, 11, 5, 6, 0.5, True, False, True),
        (6, TOPK, 4, 9, 4, 5, 1.0, False, True, False),
        (4, SWITCH, 1, 10, 5, 4, 0.5, True, True, True),
        (2, TOPK, 1, 8, 3, 7, 2.0, True, False, False),
    ]
    rng = np.random.default_rng(190)
    for n, (E, mode, k, T, d, d_ff, cf, noisy, rb, biases) in enumerate(layers):
        inp, dy = _grad_case(200 + n, T, d, E, d_ff, k, cf, mode, noisy, router_bias=rb,
                             biases=biases)
        w = tuple(float(v) for v in rng.uniform(0.2, 1.0, 3))
        _finite_difference_check(orc, inp, dy, w, 6, 210 + n)

ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
