"""GPU parity of the threshold-mask layer (moe_forward_threshold, the
inference-time gate of strictly balanced gating in "Outrageously Large Neural
Networks": expert i takes token x iff Softmax(x W_g)_i > T_i) against the
oracle's threshold mode (bal_forward with mode_bal = 1): the mask (exact, or
an explained near-threshold entry), the picks and their renormalised gates,
and the layer output; plus exact ties (P equal to T_i is not taken), tokens
no expert takes, and a token over the caller's bound on picks."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import (FLOOR_SIGMAS, act_bits, act_to_f64, check_close, check_gate_rel,
                         dev_act, dev_f32, f32_output_floor, router_value_err)
from sparsely_gated_mixture_gb300 import binding as B
from sparsely_gated_mixture_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

# A mask entry may differ from the oracle's only where the fp32 softmax gate
# can fall on the other side of the threshold: P within this relative
# distance of T_i (the fp32 router's logits carry ~1e-6 of error, which moves
# P by about twice that relative to itself).
NEAR = 1e-5


def _unpack(words: np.ndarray, E: int) -> np.ndarray:
    T = words.shape[0]
    bits = (words[:, :, None].astype(np.uint64) >> np.arange(32, dtype=np.uint64)) & 1
    return bits.reshape(T, -1)[:, :E].astype(np.uint8)


def run_threshold(w, inp, thr, kmax):
    cfg = B.config(w.T, w.d, w.E, w.d_ff, kmax, 1.0,
                   act_dtype=B.MOE_BF16 if w.dtype == "bf16" else B.MOE_F32)
    act = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    x = dev_act(inp["x"], w.dtype)
    y = torch.empty((w.T, w.d), dtype=act, device="cuda")
    idx = torch.full((w.T, kmax), -7, dtype=torch.int32, device="cuda")
    gate = torch.full((w.T, kmax), -7.0, dtype=torch.float32, device="cuda")
    words = torch.zeros((w.T, (w.E + 31) // 32), dtype=torch.int32, device="cuda")
    ws = torch.zeros(B.moe_threshold_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    B.moe_forward_threshold(cfg, x, dev_f32(inp["Wg"]), dev_f32(inp["bias"]), dev_f32(thr),
                            dev_act(inp["W1"], w.dtype), dev_act(inp["b1"], w.dtype),
                            dev_act(inp["W2"], w.dtype), dev_act(inp["b2"], w.dtype), y, ws,
                            idx, gate, words)
    st, det = B.moe_last_device_status(ws)
    return dict(status=st, detail=det, y=y, idx=idx.cpu().numpy(), gate=gate.cpu().numpy(),
                mask=_unpack(words.cpu().numpy().view(np.uint32), w.E))


def check_threshold(w, inp, thr, kmax, tokens):
    res = run_threshold(w, inp, thr, kmax)
    assert res["status"] == 0, (B.STATUS_NAMES[res["status"]], res["detail"])
    ref = oracle.bal_forward(dict(inp, mode_bal=1, thr=thr), tokens=tokens)
    P = ref["P"]
    th = thr.astype(np.float64)[None, :]
    diff = res["mask"] != ref["mask"]
    near = np.abs(P - th) <= NEAR * np.maximum(P, th)
    assert not np.any(diff & ~near), f"mask differs away from the thresholds at {np.argwhere(diff & ~near)[:5]}"
    used = res["mask"].astype(np.float64)  # the GPU's picks (oracle's, up to near-threshold entries)
    # The picks listed in expert order, then E; their gates P / S, then 0.
    T, E = w.T, w.E
    npick = used.sum(axis=1).astype(int)
    assert npick.max() <= kmax
    for t in range(T):
        picks = np.nonzero(used[t])[0]
        assert np.array_equal(res["idx"][t, :npick[t]], picks), t
        assert np.all(res["idx"][t, npick[t]:] == E), t
        assert np.all(res["gate"][t, npick[t]:] == 0.0), t
    S = (P * used).sum(axis=1, keepdims=True)
    g_dense = np.where(used == 1, P / np.where(S > 0, S, 1.0), 0.0)
    rows = np.repeat(np.arange(T), npick)
    cols = np.concatenate([np.nonzero(used[t])[0] for t in range(T)]) if npick.sum() else \
        np.zeros(0, int)
    got_g = np.concatenate([res["gate"][t, :npick[t]] for t in range(T)]) if npick.sum() else \
        np.zeros(0)
    g_rel = check_gate_rel(got_g, g_dense[rows, cols], "threshold gate") if got_g.size else 0.0
    # The output for the GPU's picks.
    idx_all = np.tile(np.arange(E, dtype=np.int32), (T, 1))
    y_ref, bad = oracle.layer_out(inp["x"], idx_all, g_dense, used.astype(np.uint8), inp["W1"],
                                  inp["W2"], inp["b1"], inp["b2"], tokens)
    assert not bad
    yg = act_to_f64(res["y"][torch.as_tensor(tokens, device="cuda").long()])
    floor = None
    if w.dtype == "f32":
        floor = f32_output_floor(inp["x"][tokens], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                                 idx_all[tokens], g_dense[tokens], used[tokens].astype(np.uint8),
                                 g_rel)
    err = check_close(yg, y_ref, w.dtype, "threshold layer output", floor)
    # Tokens no expert takes keep their input bit for bit.
    none = np.nonzero(npick == 0)[0]
    if none.size:
        sel = torch.as_tensor(none, device="cuda").long()
        xb = inp["x"][none].view(np.int16) if w.dtype == "bf16" else inp["x"][none].view(np.int32)
        assert np.array_equal(act_bits(res["y"][sel]), xb), "a token with no pick changed"
    return dict(near=int((diff & near).sum()), none=int(none.size), picks=float(npick.mean()),
                y_err=err)


def _w(name, T, d, E, d_ff, dtype="bf16"):
    return wl.Workload(name, T=T, d=d, E=E, d_ff=d_ff, k=1, cf=1.0, mode=wl.TOPK, dtype=dtype,
                       noisy=False)


# name: (workload, thresholds as multiples of 1/E (low, high), bound on picks)
CASES = {
    "thr_e8_k8": (_w("thr_e8_k8", 333, 128, 8, 64), (0.5, 1.5), 8),
    "thr_e16_k4": (_w("thr_e16_k4", 400, 64, 16, 128), (3.3, 4.5), 4),
    "thr_e64_k16": (_w("thr_e64_k16", 300, 64, 64, 64), (4.0, 6.4), 16),
    "thr_ragged_f32": (_w("thr_ragged_f32", 129, 36, 7, 50, "f32"), (0.6, 1.4), 7),
    "thr_d72": (_w("thr_d72", 200, 72, 5, 200), (0.7, 1.3), 5),
    "thr_single_token": (_w("thr_single_token", 1, 64, 8, 64), (0.5, 1.5), 8),
    "thr_e100_k16": (_w("thr_e100_k16", 257, 64, 100, 64), (6.25, 9.0), 16),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_threshold_small_parity(name):
    w, (lo, hi), kmax = CASES[name]
    inp = wl.generate(w, seed=97, biases=True)
    inp["bias"] = (np.random.default_rng(3).standard_normal(w.E) * 0.3).astype(np.float32)
    thr = (np.random.default_rng(4).uniform(lo, hi, w.E) / w.E).astype(np.float32)
    rep = check_threshold(w, inp, thr, kmax, np.arange(w.T, dtype=np.int32))
    print(name, rep)


def test_threshold_exact_ties_and_empty_tokens():
    """A zero router and no bias: every P is exactly 1/8 on both sides. T_i =
    1/8 (equal: not taken) for even experts and just below for odd ones, so
    every token takes the four odd experts with gates exactly 1/4; then every
    T_i = 1/8, so no token takes any expert and y = x bit for bit."""
    w = _w("thr_ties", 200, 64, 8, 64)
    inp = wl.generate(w, seed=99, biases=True)
    inp["Wg"] = np.zeros_like(inp["Wg"])
    thr = np.where(np.arange(8) % 2 == 0, 0.125, np.nextafter(np.float32(0.125), 0)).astype(
        np.float32)
    rep = check_threshold(w, inp, thr, 8, np.arange(w.T, dtype=np.int32))
    assert rep["near"] == 0 and rep["picks"] == 4.0
    res = run_threshold(w, inp, thr, 8)
    assert np.all(res["gate"][:, :4] == 0.25) and np.all(res["idx"][:, :4] == [1, 3, 5, 7])
    none = np.full(8, 0.125, np.float32)
    rep = check_threshold(w, inp, none, 8, np.arange(w.T, dtype=np.int32))
    assert rep["none"] == w.T


def test_threshold_over_the_bound_is_reported():
    """Thresholds every P passes with a bound of 2 picks: the first token over
    it is reported as MOE_ERR_BOUNDS and only two picks per token are kept."""
    w = _w("thr_over", 100, 64, 8, 64)
    inp = wl.generate(w, seed=98)
    res = run_threshold(w, inp, np.full(8, 1e-6, np.float32), 2)
    assert res["status"] == 6
    assert 0 <= res["detail"] < w.T
    assert np.array_equal(res["idx"], np.tile([0, 1], (w.T, 1)))


@pytest.mark.parametrize("name", sorted(wl.THR_WORKLOADS))
def test_threshold_full_size_sampled(name):
    """The benchmark's threshold layer at full size: the whole mask and every
    pick's gate, and sampled output rows."""
    w = wl.THR_WORKLOADS[name]
    inp = wl.generate(w, seed=0)
    thr = wl.thresholds(w)
    rng = np.random.default_rng(8)
    tokens = np.array(sorted(set(rng.choice(w.T, 128, replace=False).tolist()) | {0, w.T - 1}),
                      np.int32)
    rep = check_threshold(w, inp, thr, w.k, tokens)
    print(name, rep)
