"""The expert FFN stage alone (moe_expert_ffn through the C ABI) against numpy
on hand-built packed rows: ragged experts (one empty, one spanning several
128-row tiles), an N tail that is not a multiple of the 256-column tile, and
non-zero biases; the library's kernel choice, and each of the one-CTA and
CTA-pair kernels forced. A kernel-level check that localises GEMM faults; the
layer's parity against the oracle is tested in test_gpu_parity.py."""
import numpy as np
import pytest
import torch

from sparsely_gated_mixture_gb300 import binding as B
from sparsely_gated_mixture_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bf16(a):
    return wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(a))


# Row counts around the 256-row tiles of the CTA-pair kernel: an expert's
# last tile with at most 128 rows runs at M = 128 (64 rows per CTA), with
# 129 or more at M = 256; both, and the 128 / 129 and 256 / 257 boundaries.
PAIR_TAILS = [[40, 0, 296, 128, 129, 384, 1], [256, 257, 511, 64]]


SHAPES = [([130, 0, 257], 128, 320), ([1, 128, 64], 64, 64), ([300, 5], 256, 512),
          (PAIR_TAILS[0], 128, 320), (PAIR_TAILS[1], 192, 256)]


@pytest.mark.parametrize("variant", ["", "single", "pair"])
@pytest.mark.parametrize("rows,d,d_ff", SHAPES)
def test_expert_ffn_against_numpy(rows, d, d_ff, variant, monkeypatch):
    monkeypatch.setenv("MOE_FFN_TC_VARIANT", variant)
    rng = np.random.default_rng(3)
    E = len(rows)
    A = int(sum(rows)) + 7  # spare rows past the last expert
    T, k = A, 1
    cfg = B.config(T, d, E, d_ff, k, float(E), act_dtype=B.MOE_BF16)
    X = _bf16(rng.standard_normal((A, d)).astype(np.float32))
    W1 = _bf16((rng.standard_normal((E, d, d_ff)) / np.sqrt(d)).astype(np.float32))
    W2 = _bf16((rng.standard_normal((E, d_ff, d)) / np.sqrt(d_ff)).astype(np.float32))
    b1 = _bf16((0.1 * rng.standard_normal((E, d_ff))).astype(np.float32))
    b2 = _bf16((0.1 * rng.standard_normal((E, d))).astype(np.float32))
    g = rng.random(A).astype(np.float32)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    bf = lambda a: dev(a).to(torch.bfloat16)
    xbuf, w1, w2, bb1, bb2 = bf(X), bf(W1), bf(W2), bf(b1), bf(b2)
    hbuf = torch.zeros((A, d_ff), dtype=torch.bfloat16, device="cuda")
    zbuf = torch.zeros((A, d), dtype=torch.float32, device="cuda")
    ws = torch.zeros(B.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    B.moe_expert_ffn(cfg, xbuf, dev(off), dev(g), w1, bb1, w2, bb2, hbuf, zbuf, ws)
    st, det = B.moe_last_device_status(ws)
    assert st == 0, (st, det)
    H = hbuf.float().cpu().numpy().astype(np.float64)
    Z = zbuf.cpu().numpy().astype(np.float64)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        Xe = X[r0:r1].astype(np.float64)
        Href = np.maximum(Xe @ W1[e].astype(np.float64) + b1[e], 0.0)
        err = np.abs(H[r0:r1] - Href)
        assert np.all(err <= 8e-3 * (1 + np.abs(Href))), f"layer 1 expert {e}: {err.max():.3e}"
        Zref = g[r0:r1, None] * (H[r0:r1] @ W2[e].astype(np.float64) + b2[e])
        err = np.abs(Z[r0:r1] - Zref)
        assert np.all(err <= 1e-3 * (1 + np.abs(Zref))), f"layer 2 expert {e}: {err.max():.3e}"


@pytest.mark.parametrize("rows,d,d_ff", SHAPES)
def test_pair_kernel_k_backwards(rows, d, d_ff, monkeypatch):
    """The CTA-pair kernel with every tile walking K from its last block
    (MOE_FFN_SNAKE=all). By default only the odd waves of tiles do, which
    these small layers (fewer tiles than pairs) never reach; the full-size
    layers of test_gpu_parity.py run both directions."""
    monkeypatch.setenv("MOE_FFN_SNAKE", "all")
    test_expert_ffn_against_numpy(rows, d, d_ff, "pair", monkeypatch)
