"""The seeded input generator: determinism, shapes and the bf16 rounding."""
import numpy as np
import torch

from sparsely_gated_mixture_gb300 import workloads as wl


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.standard_normal(10000).astype(np.float32),
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -0.0, 65504.0], np.float32)])
    ours = wl.f32_to_bf16_bits(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = wl.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(a).to(torch.bfloat16).float().numpy())


def test_generate_deterministic_and_shaped():
    w = wl.WORKLOADS["noisy_top4_e16"].with_(T=64)
    a = wl.generate(w, seed=3)
    b = wl.generate(w, seed=3)
    for key in ("x", "Wg", "Wn", "noise", "W1", "W2"):
        assert np.array_equal(a[key], b[key])
    assert a["x"].shape == (64, 512) and a["x"].dtype == np.uint16
    assert a["Wg"].dtype == np.float32 and a["Wg"].shape == (512, 16)
    assert a["W1"].shape == (16, 512, 1024) and a["W2"].shape == (16, 1024, 512)
    assert a["b1"] is None and a["bias"] is None
    c = wl.generate(w, seed=4)
    assert not np.array_equal(a["x"], c["x"])


def test_capacities_of_the_workloads():
    want = {"switch_top1_toy": 2, "noisy_top4_e16": 2048, "switch_top1_zipf_e64": 320,
            "top2_large_experts": 2560, "many_small_experts_e1024": 192}
    for name, C in want.items():
        assert wl.WORKLOADS[name].capacity == C


def test_zipf_bias():
    w = wl.WORKLOADS["switch_top1_zipf_e64"].with_(T=16, d=8, d_ff=8)
    b = wl.generate(w)["bias"]
    assert b[0] == 0.0 and np.all(np.diff(b) < 0)
    np.testing.assert_allclose(b[9], 1.5 * np.log(1 / 10), rtol=1e-6)
