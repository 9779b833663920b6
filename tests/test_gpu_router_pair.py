"""The tensor-core router's CTA-pair form (two SMs per 256-token tile, for
many column blocks) against the fp64 oracle, and against the one-CTA form on
the same inputs ("Outrageously Large Neural Networks", Noisy Top-K Gating,
Eq. 4). MOE_ROUTER_PAIR=1 selects the pair form wherever it applies, =0 the
one-CTA form; the full-size many-small-experts layer takes the pair form by
default and is covered by test_gpu_parity.py.

The cases are ragged on purpose: token counts that leave the odd CTA of the
last pair with few or no rows, a width that is not a whole number of 64-deep
K steps, and an expert count whose last column block is partial."""
import numpy as np
import pytest

from test_gpu_parity import check_stages
from sparsely_gated_mixture_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CASES = {
    # 900 = 3 * 256 + 132: the last pair's odd CTA holds 4 tokens
    "e1024_t900": wl.WORKLOADS["many_small_experts_e1024"].with_(T=900),
    # K tail (200 = 3 * 64 + 8); 2E = 192 columns: three column blocks
    "ragged_k_e96": wl.Workload("ragged_k_e96", T=333, d=200, E=96, d_ff=64, k=4, cf=1.0,
                                mode=wl.TOPK, dtype="bf16", noisy=True),
    # no noise: 200 columns, the last block 8 wide; Switch gate
    "clean_switch_e200": wl.Workload("clean_switch_e200", T=517, d=128, E=200, d_ff=64, k=1,
                                     cf=1.25, mode=wl.SWITCH, dtype="bf16", noisy=False),
    # one token: the odd CTA's rows are all past T
    "single_token_e96": wl.Workload("single_token_e96", T=1, d=64, E=96, d_ff=64, k=2, cf=1.0,
                                    mode=wl.TOPK, dtype="bf16", noisy=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_pair_router_matches_oracle_and_one_cta_form(name, monkeypatch):
    w = CASES[name]
    inp = wl.generate(w, seed=23, biases=True)
    monkeypatch.setenv("MOE_ROUTER_PAIR", "1")
    pair, _ = check_stages(w, inp)
    monkeypatch.setenv("MOE_ROUTER_PAIR", "0")
    one, _ = check_stages(w, inp)
    # Both forms add the same bf16 products in the same K order per output;
    # the selections and thresholds agree exactly.
    assert np.array_equal(pair["idx"], one["idx"])
    assert np.array_equal(pair["thr"], one["thr"])
    assert np.array_equal(pair["gate"], one["gate"])
    assert np.array_equal(pair["out3"], one["out3"])
