"""GPU parity: the CUDA path, called through the C ABI, against the fp64 oracle
on the same seeded inputs.

Small cases span several tiles and a ragged tail and are compared element by
element; the five measured workloads at full size (the configuration the
benchmark times) are compared on every index, slot and balancing value and on
sampled output rows.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import (FLOOR_SIGMAS, F32_RTOL, TIE_TOL, act_bits, act_to_f64, check_close,
                         check_gate_rel, check_rel, f32_output_floor, oracle_gate,
                         reconcile_selection, router_value_err, run_forward, run_stages,
                         to_device)
from sparsely_gated_mixture_gb300 import binding as B
from sparsely_gated_mixture_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

W = wl.WORKLOADS


def _compare(w, inp, res, ref_gate, tokens, report):
    """Checks shared by the stage-wise and forward runs. Returns the
    reconciled selection for reuse."""
    T, k, E = w.T, w.k, w.E
    used, ties, bad = reconcile_selection(ref_gate["H"], ref_gate["idx"], res["idx"])
    assert not bad, f"expert choices differ beyond near-ties at tokens {bad[:10]}"
    report["ties"] = ties
    mode = int(inp["mode"])
    g_ref = oracle.gates_given(ref_gate["H"], used, mode)
    g_rel = check_gate_rel(res["gate"], g_ref)
    report["gate_max_rel"] = g_rel
    C = oracle.capacity(T, E, k, w.cf, w.min_cap)
    pos, keep, count = oracle.slots(used, E, C)
    assert np.array_equal(res["pos"], pos), "slot positions differ"
    assert np.array_equal(res["keep"], keep), "drop masks differ"
    # Output rows: the oracle's per-token loop over accepted experts.
    y_ref, bad_y = oracle.layer_out(inp["x"], used, g_ref, keep, inp["W1"], inp["W2"], inp["b1"],
                                    inp["b2"], tokens)
    assert not bad_y
    y = act_to_f64(res["y"][torch.as_tensor(tokens, device="cuda").long()])
    floor = None
    if w.dtype == "f32":
        floor = f32_output_floor(inp["x"][tokens], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                                 used[tokens], g_ref[tokens], keep[tokens], g_rel)
    report["y_max_err"] = check_close(y, y_ref, w.dtype, "layer output y", floor)
    # Tokens with every choice dropped come out bit-identical to their input.
    drop = np.nonzero(~keep.astype(bool).any(axis=1))[0]
    report["dropped_tokens"] = int(drop.size)
    if drop.size:
        dsel = torch.as_tensor(drop, device="cuda").long()
        x_bits = inp["x"][drop].view(np.int16) if w.dtype == "bf16" else inp["x"][drop].view(np.int32)
        assert np.array_equal(act_bits(res["y"][dsel]), x_bits), "dropped token changed"
    return used, g_ref, pos, keep, count, C


def _check_aux(w, inp, ref_gate, used, g_ref, out3, importance=None, load=None):
    ax = oracle.aux(ref_gate["c"], ref_gate["sigma"], ref_gate["H"], used, g_ref, ref_gate["hk"],
                    ref_gate["hk1"], inp["Wn"] is not None)
    check_rel(out3, ax["out3"], "aux out3 [importance CV^2, load CV^2, switch aux]")
    if importance is not None:
        check_rel(importance, ax["importance"], "importance")
        check_rel(load, ax["load"], "load")
    return ax


def check_stages(w, inp, tokens=None):
    d = to_device(w, inp)
    res = run_stages(w, d)
    assert res["status"] == 0, (B.STATUS_NAMES[res["status"]], res["detail"])
    ref_gate = oracle_gate(inp)
    if tokens is None:
        tokens = np.arange(w.T, dtype=np.int32)
    report = {}
    used, g_ref, pos, keep, count, C = _compare(w, inp, res, ref_gate, tokens, report)
    # Gate thresholds, counts, offsets.
    thr_ref = np.stack([ref_gate["hk"], ref_gate["hk1"]], axis=1)
    fin = np.isfinite(thr_ref)
    assert np.array_equal(np.isfinite(res["thr"]), fin)
    # The k-th and (k+1)-th largest H (lower index first on ties): 1e-4
    # relative, or the router's own fp32 rounding-error floor near zero.
    order = np.argsort(-ref_gate["H"], axis=1, kind="stable")
    cols = order[:, [w.k - 1, min(w.k, w.E - 1)]]
    x64 = wl.bf16_bits_to_f32(inp["x"]).astype(np.float64) if w.dtype == "bf16" else inp["x"]
    thr_floor = FLOOR_SIGMAS * router_value_err(x64, inp["Wg"], inp["Wn"], inp["noise"],
                                                inp["bias"], cols)
    lim = np.maximum(F32_RTOL * np.abs(thr_ref[fin]), thr_floor[fin])
    terr = np.abs(res["thr"][fin] - thr_ref[fin])
    assert np.all(terr <= lim), (f"gate thresholds: max err {terr.max():.3e}, worst excess "
                                 f"{(terr / lim).max():.3f} of the bound")
    report["thr_floor_used"] = int((thr_floor[fin] > F32_RTOL * np.abs(thr_ref[fin])).sum())
    assert np.array_equal(res["count"], count)
    off = np.concatenate([[0], np.cumsum(np.minimum(count, C))]).astype(np.int32)
    assert np.array_equal(res["offset"], off)
    # Dispatch: every accepted (t, j) sits at row offset[e] + pos, in token order.
    a = np.nonzero(keep.reshape(-1))[0]
    t_of, j_of = a // w.k, a % w.k
    rows = off[used.reshape(-1)[a]] + pos.reshape(-1)[a]
    assert np.array_equal(np.sort(rows), np.arange(off[-1]))
    assert np.array_equal(res["row_token"][rows], a.astype(np.int32))
    assert np.array_equal(res["row_gate"][rows], res["gate"].reshape(-1)[a])
    xb = act_bits(res["xbuf"][: off[-1]])
    x_bits = inp["x"].view(np.int16) if w.dtype == "bf16" else inp["x"].view(np.int32)
    assert np.array_equal(xb[rows], x_bits[t_of]), "gathered rows differ from their tokens"
    _check_aux(w, inp, ref_gate, used, g_ref, res["out3"], res["importance"], res["load"])
    return res, report


def check_forward(w, inp, tokens, stages=None):
    d = to_device(w, inp)
    res = run_forward(w, d)
    assert res["status"] == 0, (B.STATUS_NAMES[res["status"]], res["detail"])
    ref_gate = oracle_gate(inp)
    report = {}
    used, g_ref, *_ = _compare(w, inp, res, ref_gate, tokens, report)
    _check_aux(w, inp, ref_gate, used, g_ref, res["out3"])
    if stages is not None:
        if w.dtype == "bf16":
            # moe_forward may keep the expert outputs in bf16 where the stage
            # calls keep fp32 (one more rounding per term); both are checked
            # against the oracle above, and against each other here.
            check_close(act_to_f64(res["y"]), act_to_f64(stages["y"]), w.dtype,
                        "moe_forward against the stage calls")
        else:
            assert torch.equal(res["y"], stages["y"]), "moe_forward and the stage calls differ"
    return res, report


SMALL = {
    "toy": W["switch_top1_toy"],
    "noisy_top4_e16": W["noisy_top4_e16"].with_(T=517),
    "zipf_switch_e64": W["switch_top1_zipf_e64"].with_(T=700),
    "top2_large_dims": W["top2_large_experts"].with_(T=40),
    "top2_mid": W["top2_large_experts"].with_(T=333, d=512, d_ff=1024),
    "e1024_top4": W["many_small_experts_e1024"].with_(T=900),
    "ragged_bf16": wl.Workload("ragged_bf16", T=333, d=72, E=5, d_ff=200, k=3, cf=0.8,
                               mode=wl.TOPK, dtype="bf16", noisy=True),
    "ragged_f32": wl.Workload("ragged_f32", T=129, d=36, E=7, d_ff=50, k=2, cf=1.0,
                              mode=wl.TOPK, dtype="f32", noisy=True),
    "single_token": wl.Workload("single_token", T=1, d=64, E=4, d_ff=128, k=2, cf=1.0,
                                mode=wl.TOPK, dtype="bf16", noisy=True),
    "one_expert_dense": wl.Workload("one_expert_dense", T=130, d=64, E=1, d_ff=192, k=1, cf=1.0,
                                    mode=wl.SWITCH, dtype="bf16", noisy=False),
    "k_equals_E": wl.Workload("k_equals_E", T=257, d=128, E=4, d_ff=256, k=4, cf=1.0,
                              mode=wl.TOPK, dtype="bf16", noisy=True),
    "heavy_drop": wl.Workload("heavy_drop", T=300, d=128, E=8, d_ff=256, k=2, cf=0.05,
                              mode=wl.TOPK, dtype="bf16", noisy=True),
    "switch_f32_noisy": wl.Workload("switch_f32_noisy", T=200, d=24, E=6, d_ff=40, k=1, cf=1.1,
                                    mode=wl.SWITCH, dtype="f32", noisy=True),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_parity(name):
    w = SMALL[name]
    inp = wl.generate(w, seed=11, biases=name not in ("toy",))
    stages, rep = check_stages(w, inp)
    check_forward(w, inp, np.arange(w.T, dtype=np.int32), stages)


def test_toy_zero_bias_exact_workload():
    """The Switch toy exactly as specified: seed 0, zero biases, no noise."""
    w = W["switch_top1_toy"]
    inp = wl.generate(w, seed=0)
    check_stages(w, inp)


def _sample_tokens(T, n, seed):
    rng = np.random.default_rng(seed)
    s = set(rng.choice(T, size=min(n, T), replace=False).tolist()) | {0, T - 1}
    return np.array(sorted(s), dtype=np.int32)


@pytest.mark.parametrize("name", sorted(W))
def test_full_size_sampled(name):
    """Each measured workload at full size, launched as the benchmark launches
    it: every index, slot and balancing value, and sampled output rows."""
    w = W[name]
    inp = wl.generate(w, seed=0)
    tokens = _sample_tokens(w.T, 48 if w.d * w.d_ff > 10**7 else 256, seed=1)
    res, rep = check_forward(w, inp, tokens)
    print(name, "near-ties:", len(rep["ties"]), "dropped:", rep["dropped_tokens"],
          "y max err:", rep["y_max_err"])


def test_deterministic():
    w = SMALL["noisy_top4_e16"]
    inp = wl.generate(w, seed=5)
    d = to_device(w, inp)
    a = run_forward(w, d)
    b = run_forward(w, d)
    assert torch.equal(a["y"], b["y"])
    assert np.array_equal(a["out3"], b["out3"])
    assert np.array_equal(a["pos"], b["pos"])


def test_nonfinite_input_reported():
    w = SMALL["top2_mid"]
    inp = wl.generate(w, seed=6)
    inp["x"] = inp["x"].copy()
    inp["x"][5, 3] = 0x7FC0  # bf16 NaN
    d = to_device(w, inp)
    res = run_forward(w, d)
    assert res["status"] == 4  # MOE_ERR_NONFINITE


def test_bad_arguments_rejected_before_launch():
    w = SMALL["top2_mid"]
    cfg = B.config_for(w)
    bad = B.config_for(w.with_(k=9))  # k > E
    with pytest.raises(B.MoEError) as e:
        B.moe_workspace_size(bad)
    assert e.value.status == 1
    inp = wl.generate(w, seed=7)
    d = to_device(w, inp)
    ws = torch.empty(B.moe_workspace_size(cfg) + 256, dtype=torch.uint8, device="cuda")
    y = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.MoEError) as e:  # misaligned workspace
        B.moe_forward(cfg, d["x"], d["Wg"], d["Wn"], d["noise"], None, d["W1"], None, d["W2"],
                      None, y, None, ws.data_ptr() + 8)
    assert e.value.status == 1
    with pytest.raises(B.MoEError):  # noise weights without noise
        B.moe_forward(cfg, d["x"], d["Wg"], d["Wn"], None, None, d["W1"], None, d["W2"], None, y,
                      None, ws)


WIDE = {
    # E = 301: one expert per thread in the column sums, 16 values per lane in
    # the selection; k = 5 takes the long chosen-list form.
    "e301_k5": wl.Workload("e301_k5", T=333, d=64, E=301, d_ff=64, k=5, cf=1.0, mode=wl.TOPK,
                           dtype="bf16", noisy=True),
    "e1024_switch": wl.Workload("e1024_switch", T=300, d=128, E=1024, d_ff=64, k=1, cf=1.0,
                                mode=wl.SWITCH, dtype="bf16", noisy=False),
}


@pytest.mark.parametrize("name", sorted(WIDE))
def test_wide_router_parity(name):
    w = WIDE[name]
    inp = wl.generate(w, seed=13, biases=True)
    stages, _ = check_stages(w, inp)
    check_forward(w, inp, np.arange(w.T, dtype=np.int32), stages)


@pytest.mark.parametrize("levels", [0, 3])
def test_tied_logits_wide(levels):
    """Exact ties in wide rows: a zero clean router with a bias on a coarse
    grid, so every token's logits are the bias. levels = 0 ties all 1024
    experts (more candidates than a warp holds); levels = 3 leaves a few
    dozen experts tied at the top. Ties are broken by the lower index on both
    sides, so the choices must match exactly."""
    w = wl.Workload("tied_e1024", T=200, d=64, E=1024, d_ff=64, k=4, cf=2.0, mode=wl.TOPK,
                    dtype="bf16", noisy=False)
    inp = wl.generate(w, seed=17)
    inp["Wg"] = np.zeros_like(inp["Wg"])
    rng = np.random.default_rng(3)
    inp["bias"] = (np.round(rng.standard_normal(w.E) * levels) if levels else
                   np.zeros(w.E)).astype(np.float32)
    res, _ = check_stages(w, inp)
    ref = oracle_gate(inp)
    assert np.array_equal(res["idx"], ref["idx"])


CLEAN_TOPK = {
    # Top-k without the noise term: the router writes H alone, the load sum is
    # the pre-capacity count; E = 32 takes the fused selection, E = 512 the
    # column sums.
    "clean_top2_e32": wl.Workload("clean_top2_e32", T=300, d=128, E=32, d_ff=64, k=2, cf=1.0,
                                  mode=wl.TOPK, dtype="bf16", noisy=False),
    "clean_top3_e512": wl.Workload("clean_top3_e512", T=300, d=64, E=512, d_ff=64, k=3,
                                   cf=1.5, mode=wl.TOPK, dtype="bf16", noisy=False),
}


@pytest.mark.parametrize("name", sorted(CLEAN_TOPK))
def test_clean_topk_parity(name):
    w = CLEAN_TOPK[name]
    inp = wl.generate(w, seed=23, biases=True)
    stages, _ = check_stages(w, inp)
    check_forward(w, inp, np.arange(w.T, dtype=np.int32), stages)


@pytest.mark.parametrize("E", [64, 512])
def test_router_bias_with_noise(E):
    """A router logit bias together with the noise term (c = x Wg + b, then
    H = c + n sigma), on the fused (E = 64) and column (E = 512) paths."""
    w = wl.Workload(f"noisy_bias_e{E}", T=400, d=128, E=E, d_ff=64, k=2, cf=1.25, mode=wl.TOPK,
                    dtype="bf16", noisy=True)
    inp = wl.generate(w, seed=29, biases=True)
    inp["bias"] = (np.random.default_rng(5).standard_normal(E) * 0.5).astype(np.float32)
    stages, _ = check_stages(w, inp)
    check_forward(w, inp, np.arange(w.T, dtype=np.int32), stages)


FUSED = {
    # The tensor-core router selects in its own epilogue when every expert of
    # a token sits in one 64-column block (E <= 32 with the noise term, 64
    # without) and k <= 8: the longest pick lists, k = E, and a grid of more
    # row blocks than SMs (one tile per CTA, several waves).
    "fused_noisy_e32_k5": wl.Workload("fused_noisy_e32_k5", T=300, d=128, E=32, d_ff=64, k=5,
                                      cf=1.0, mode=wl.TOPK, dtype="bf16", noisy=True),
    "fused_clean_e64_k8": wl.Workload("fused_clean_e64_k8", T=257, d=64, E=64, d_ff=64, k=8,
                                      cf=1.25, mode=wl.TOPK, dtype="bf16", noisy=False),
    "fused_k_equals_E8": wl.Workload("fused_k_equals_E8", T=200, d=64, E=8, d_ff=64, k=8, cf=1.0,
                                     mode=wl.TOPK, dtype="bf16", noisy=True),
    "fused_switch_noisy_e16": wl.Workload("fused_switch_noisy_e16", T=333, d=96, E=16, d_ff=64,
                                          k=1, cf=1.0, mode=wl.SWITCH, dtype="bf16", noisy=True),
}


@pytest.mark.parametrize("name", sorted(FUSED))
def test_fused_selection_parity(name):
    w = FUSED[name]
    inp = wl.generate(w, seed=31, biases=True)
    stages, _ = check_stages(w, inp)
    check_forward(w, inp, np.arange(w.T, dtype=np.int32), stages)


def test_fused_selection_many_waves():
    """153 row blocks of 128 tokens (one more than the SMs), the last ragged:
    every index, slot and balancing value, and sampled rows."""
    w = wl.Workload("fused_waves", T=152 * 128 + 77, d=64, E=8, d_ff=64, k=2, cf=1.25,
                    mode=wl.TOPK, dtype="bf16", noisy=True)
    inp = wl.generate(w, seed=37, biases=True)
    tokens = _sample_tokens(w.T, 512, seed=2)
    check_stages(w, inp, tokens)
    check_forward(w, inp, tokens)


@pytest.mark.parametrize("E,levels", [(16, 0), (16, 2), (64, 0), (64, 3)])
def test_tied_logits_fused(E, levels):
    """Exact ties on the fused selection: a zero clean router with a bias on a
    coarse grid (levels = 0: every expert tied), so the picks, thresholds and
    gates must match the oracle's lower-index-first order exactly."""
    w = wl.Workload(f"tied_fused_e{E}", T=200, d=64, E=E, d_ff=64, k=4, cf=2.0, mode=wl.TOPK,
                    dtype="bf16", noisy=False)
    inp = wl.generate(w, seed=19)
    inp["Wg"] = np.zeros_like(inp["Wg"])
    rng = np.random.default_rng(4)
    inp["bias"] = (np.round(rng.standard_normal(w.E) * levels) if levels else
                   np.zeros(w.E)).astype(np.float32)
    res, _ = check_stages(w, inp)
    ref = oracle_gate(inp)
    assert np.array_equal(res["idx"], ref["idx"])
