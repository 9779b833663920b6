"""GPU parity of the hierarchical layer (moe_forward_hier) against the fp64
oracle: choices (exact, or explained near-ties at either gate level), product
gates, slots, output rows and the two hierarchical losses."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import (act_bits, act_to_f64, check_close, check_gate_rel, check_rel,
                         f32_output_floor, hier_given, hier_to_device, reconcile_hier,
                         run_hier_forward)
from sparsely_gated_mixture_gb300 import binding as B
from sparsely_gated_mixture_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

HW = wl.HierWorkload


def check_hier(w, inp, tokens):
    d = hier_to_device(w, inp)
    res = run_hier_forward(w, d)
    assert res["status"] == 0, (B.STATUS_NAMES[res["status"]], res["detail"])
    ref = oracle.hier_forward(inp, tokens=tokens)
    used, ties, bad = reconcile_hier(ref, res["idx"], w.a, w.b, w.kp, w.ks)
    assert not bad, f"choices differ beyond near-ties at tokens {bad[:10]}"
    g = hier_given(inp, ref, used, w, tokens)
    g_rel = check_gate_rel(res["gate"], g["gate"], "product gate")
    assert np.array_equal(res["pos"], g["pos"]), "slot positions differ"
    assert np.array_equal(res["keep"], g["keep"]), "drop masks differ"
    y = act_to_f64(res["y"][torch.as_tensor(tokens, device="cuda").long()])
    floor = None
    if w.dtype == "f32":
        floor = f32_output_floor(inp["x"][tokens], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                                 used[tokens], g["gate"][tokens], g["keep"][tokens], g_rel)
    y_err = check_close(y, g["y"], w.dtype, "hierarchical layer output y_H", floor)
    drop = np.nonzero(~g["keep"].astype(bool).any(axis=1))[0]
    if drop.size:
        dsel = torch.as_tensor(drop, device="cuda").long()
        x_bits = inp["x"][drop].view(np.int16) if w.dtype == "bf16" else inp["x"][drop].view(
            np.int32)
        assert np.array_equal(act_bits(res["y"][dsel]), x_bits), "dropped token changed"
    check_rel(res["out2"], g["out2"], "[CV(Importance_H)^2, CV(Load_H)^2]")
    return dict(ties=ties, y_err=y_err, dropped=int(drop.size), group_count=g["count"])


SMALL = {
    "hier_4x8": HW("hier_4x8", T=333, d=128, a=4, b=8, kp=2, ks=2, d_ff=64, cf=1.0,
                   dtype="bf16", noisy=True),
    "hier_one_group": HW("hier_one_group", T=257, d=64, a=1, b=16, kp=1, ks=4, d_ff=64, cf=1.25,
                         dtype="bf16", noisy=True),
    "hier_wide_groups_b100": HW("hier_wide_groups_b100", T=200, d=64, a=3, b=100, kp=2, ks=3,
                                d_ff=64, cf=1.5, dtype="bf16", noisy=True),
    "hier_clean_8x8": HW("hier_clean_8x8", T=300, d=96, a=8, b=8, kp=2, ks=1, d_ff=64, cf=1.0,
                         dtype="bf16", noisy=False),
    "hier_ks_equals_b": HW("hier_ks_equals_b", T=150, d=64, a=6, b=2, kp=3, ks=2, d_ff=64,
                           cf=1.0, dtype="bf16", noisy=True),
    "hier_f32": HW("hier_f32", T=129, d=36, a=5, b=3, kp=2, ks=2, d_ff=50, cf=1.0, dtype="f32",
                   noisy=True),
}


EDGE = {
    # one token; the largest k (k_p * k_s = 16); noise on the primary gate
    # only is covered by hier_clean_8x8's counterpart below
    "hier_single_token": HW("hier_single_token", T=1, d=64, a=4, b=8, kp=2, ks=2, d_ff=64,
                            cf=1.0, dtype="bf16", noisy=True),
    "hier_k16": HW("hier_k16", T=200, d=64, a=8, b=16, kp=4, ks=4, d_ff=64, cf=1.0,
                   dtype="bf16", noisy=True),
    "hier_kp_equals_a": HW("hier_kp_equals_a", T=150, d=64, a=3, b=8, kp=3, ks=2, d_ff=64,
                           cf=1.0, dtype="bf16", noisy=True),
    # the grouped secondary router without noise (16 columns per group), and
    # with a group spanning three 64-column blocks
    "hier_grouped_clean_b16": HW("hier_grouped_clean_b16", T=300, d=64, a=6, b=16, kp=2, ks=3,
                                 d_ff=64, cf=1.0, dtype="bf16", noisy=False),
    "hier_grouped_b96": HW("hier_grouped_b96", T=400, d=128, a=4, b=96, kp=2, ks=4, d_ff=64,
                           cf=1.25, dtype="bf16", noisy=True),
}
SMALL.update(EDGE)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_hier_small_parity(name):
    w = SMALL[name]
    inp = wl.generate_hier(w, seed=61, biases=True)
    check_hier(w, inp, np.arange(w.T, dtype=np.int32))


def test_hier_empty_group():
    """A group no token's primary gate picks: |X^(i)| = 0 and its Load_H
    entries are 0, on the GPU as in the oracle."""
    w = HW("hier_empty", T=200, d=64, a=4, b=8, kp=2, ks=2, d_ff=64, cf=2.0, dtype="bf16",
           noisy=False)
    inp = wl.generate_hier(w, seed=67)
    Wp = np.zeros_like(inp["Wp"])
    x = wl.bf16_bits_to_f32(inp["x"]).copy()
    x[:, 0] = 1.0
    inp["x"] = wl.f32_to_bf16_bits(x)
    Wp[0] = [3.0, 2.0, 1.0, -8.0]
    inp["Wp"] = Wp
    rep = check_hier(w, inp, np.arange(w.T, dtype=np.int32))
    assert rep["group_count"][3] == 0


def _sample(T, n, seed):
    rng = np.random.default_rng(seed)
    s = set(rng.choice(T, size=min(n, T), replace=False).tolist()) | {0, T - 1}
    return np.array(sorted(s), dtype=np.int32)


@pytest.mark.parametrize("name", sorted(wl.HIER_WORKLOADS))
def test_hier_full_size_sampled(name):
    """The measured hierarchical workload at full size: every choice, slot and
    loss, and sampled output rows."""
    w = wl.HIER_WORKLOADS[name]
    inp = wl.generate_hier(w, seed=0)
    rep = check_hier(w, inp, _sample(w.T, 256, seed=3))
    print(name, "near-ties:", len(rep["ties"]), "dropped:", rep["dropped"], "y max err:",
          rep["y_err"])
