"""The device normal CDF of the load estimator (Phi in P(x, i), "Outrageously
Large Neural Networks", Eq. 9), evaluated through moe_eval_normal_cdf on a
dense grid, against the exact Phi(u) = erfc(-u / sqrt 2) / 2 in fp64 (the
standard library's erfc), with CUDA's own fp32 erfcf (through torch) beside
it for comparison."""
import math

import numpy as np
import pytest
import torch

from sparsely_gated_mixture_gb300 import binding as B

pytestmark = pytest.mark.gpu


def test_normal_cdf_against_erfc_grid():
    u = np.concatenate([np.linspace(-14.0, 14.0, 400001),
                        np.random.default_rng(0).standard_normal(100000) * 3.0])
    u32 = u.astype(np.float32)
    exact = np.array([0.5 * math.erfc(-float(v) / math.sqrt(2.0)) for v in u32], np.float64)
    ut = torch.from_numpy(u32).cuda()
    out = torch.empty_like(ut)
    B.moe_eval_normal_cdf(ut, out)
    got = out.cpu().numpy().astype(np.float64)
    cuda_erfc = (0.5 * torch.special.erfc(-ut * np.float32(1.0 / math.sqrt(2.0)))).cpu().numpy()
    # Where Phi >= 1e-7 (z = |u|/sqrt 2 <= 3.7): relative error within 3e-6,
    # the sum of the worst cases of each step: the fit itself 1.2e-7; the
    # division for t 2 ulp (2.4e-7, also carried through P(t)); Horner's nine
    # FMAs on P about 3.6e-7 absolute; the exponent (P - z^2) - e, |.| <= 14,
    # rounded once (8.4e-7 absolute); the fast exponential scaling it by
    # log2(e) in fp32 (1.2e-6 absolute in the power of 2, 8.3e-7 relative)
    # and its own 2e-7; the final products 1.2e-7. Below 1e-7, absolute
    # 1e-12 (such P are far under the 1e-4 tolerance of any load sum).
    big = exact >= 1e-7
    rel = np.abs(got[big] - exact[big]) / exact[big]
    assert rel.max() <= 3e-6, f"max relative error {rel.max():.3e} at u = {u32[big][rel.argmax()]}"
    small = ~big
    assert np.all(np.abs(got[small] - exact[small]) <= 1e-12)
    assert np.all((got >= 0.0) & (got <= 1.0))
    assert np.all(np.diff(got[:400001]) >= -1e-7), "Phi must not decrease along the grid"
    rel_cuda = np.abs(cuda_erfc[big] - exact[big]) / exact[big]
    print(f"max relative error where Phi >= 1e-7: library {rel.max():.3e}, "
          f"CUDA erfcf {rel_cuda.max():.3e}")
