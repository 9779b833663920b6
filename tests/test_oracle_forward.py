"""The oracle's whole forward path on generated inputs: invariants stated on
the pages (gates sum to 1, dropped tokens unchanged, token-order slots)."""
import numpy as np

import oracle
from sparsely_gated_mixture_gb300 import workloads as wl


def test_toy_switch_forward():
    w = wl.WORKLOADS["switch_top1_toy"]
    inp = wl.generate(w, seed=0)
    out = oracle.forward(inp)
    assert out["C"] == 2
    assert not out["nonfinite"]
    kept = out["keep"][:, 0].astype(bool)
    x = inp["x"].astype(np.float64)
    assert np.array_equal(out["y"][~kept], x[~kept])
    np.testing.assert_allclose(out["f"].sum(), 1.0)
    assert np.all(out["count"] == np.bincount(out["idx"][:, 0], minlength=3))


def test_noisy_topk_forward_small():
    w = wl.WORKLOADS["noisy_top4_e16"].with_(T=96, d=32, d_ff=48, cf=0.5)
    inp = wl.generate(w, seed=1, biases=True)
    out = oracle.forward(inp)
    np.testing.assert_allclose(out["gate"].sum(axis=1), 1.0, rtol=1e-13)
    assert out["keep"].sum() == np.minimum(out["count"], out["C"]).sum()
    full_drop = ~out["keep"].astype(bool).any(axis=1)
    x = wl.bf16_bits_to_f32(inp["x"]).astype(np.float64)
    assert np.array_equal(out["y"][full_drop], x[full_drop])
    assert abs(out["importance"].sum() - w.T) < 1e-9
