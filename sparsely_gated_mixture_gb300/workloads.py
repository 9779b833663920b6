"""Seeded synthetic inputs for the MoE layer forward path.

This module only draws random numbers and casts them; it holds none of the
layer's arithmetic, so both the CUDA path's tests and the oracle take their
inputs from here.

Recipe (the same for every workload): one PCG64 stream seeded with ``seed``,
drawn in the fixed order x, W_g, W_noise, noise, W1, b1, W2, b2:

* x ~ N(0, 1) [T, d]
* W_g, W_noise ~ N(0, 1/d) [d, E]  (fp32: the router runs in fp32)
* noise ~ N(0, 1) [T, E]           (the StandardNormal() draw of the noisy gate)
* W1 ~ N(0, 1/d) [E, d, d_ff], W2 ~ N(0, 1/d_ff) [E, d_ff, d]  (N(0, 1/fan_in))
* b1, b2 zero unless ``biases=True``, then N(0, 0.1^2)
* the Zipf-skewed workload adds a router bias b_e = 1.5 * ln(1 / (e + 1)) and
  draws W_g from N(0, 25/d) (``router_scale`` 5): that logit scale is what
  makes the stated bias send 15-25% of the tokens past capacity (about 23%);
  with N(0, 1/d) it would send about 88%.

bf16 workloads round x, W1, W2, b1, b2 from fp32 to bf16 with
round-to-nearest-even and keep the bit patterns as uint16; both sides of every
comparison receive those same bits.

The backward's upstream gradient dy ~ N(0, 1) [T, d] comes from a separate
stream (``generate_dy``), rounded like x.

Hierarchical layers (``HierWorkload``, a groups of b experts) draw, in order:
x; W_p, W_pnoise ~ N(0, 1/d) [d, a] and noise_p ~ N(0, 1) [T, a] for the
primary gate; W_s, W_snoise ~ N(0, 1/d) [d, a*b] and noise_s ~ N(0, 1)
[T, a*b] for the secondary gates (group i owns columns i*b .. i*b+b-1); then
W1, b1, W2, b2 over the a*b experts as above.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

TOPK = "topk"      # Softmax(KeepTopK(H, k))
SWITCH = "switch"  # full softmax, argmax, gate = p[argmax]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    d_ff: int
    k: int
    cf: float
    mode: str
    dtype: str          # "f32" or "bf16": x, W1, b1, W2, b2 and the output y
    noisy: bool
    zipf_bias: bool = False
    min_cap: int = 1
    router_scale: float = 1.0  # W_g ~ N(0, router_scale^2 / d)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def capacity(self) -> int:
        """Expert capacity max(min_cap, min(T, floor(k*T*cf/E))), for labels."""
        c = math.floor(self.k * self.T * self.cf / self.E)
        return max(self.min_cap, min(self.T, c))

    def expert_flops(self, accepted: int) -> int:
        """Multiply-adds x 2 of both expert layers for ``accepted`` rows."""
        return 4 * self.d * self.d_ff * accepted

    def router_flops(self) -> int:
        cols = 2 * self.E if self.noisy else self.E
        return 2 * self.T * self.d * cols


# The five workloads the layer is measured and checked on.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("switch_top1_toy", T=8, d=4, E=3, d_ff=8, k=1, cf=1.0, mode=SWITCH,
                 dtype="f32", noisy=False),
        Workload("noisy_top4_e16", T=4096, d=512, E=16, d_ff=1024, k=4, cf=2.0, mode=TOPK,
                 dtype="bf16", noisy=True),
        Workload("switch_top1_zipf_e64", T=16384, d=768, E=64, d_ff=3072, k=1, cf=1.25,
                 mode=SWITCH, dtype="bf16", noisy=False, zipf_bias=True, router_scale=5.0),
        Workload("top2_large_experts", T=8192, d=4096, E=8, d_ff=14336, k=2, cf=1.25,
                 mode=TOPK, dtype="bf16", noisy=True),
        Workload("many_small_experts_e1024", T=32768, d=512, E=1024, d_ff=1024, k=4, cf=1.5,
                 mode=TOPK, dtype="bf16", noisy=True),
    ]
}


@dataclasses.dataclass(frozen=True)
class HierWorkload:
    """A hierarchical layer: a groups of b experts, kp groups then ks experts
    in each picked group, so k = kp * ks choices per token over a*b experts."""
    name: str
    T: int
    d: int
    a: int
    b: int
    kp: int
    ks: int
    d_ff: int
    cf: float
    dtype: str
    noisy: bool
    min_cap: int = 1

    def with_(self, **kw) -> "HierWorkload":
        return dataclasses.replace(self, **kw)

    @property
    def E(self) -> int:
        return self.a * self.b

    @property
    def k(self) -> int:
        return self.kp * self.ks

    @property
    def capacity(self) -> int:
        c = math.floor(self.k * self.T * self.cf / self.E)
        return max(self.min_cap, min(self.T, c))

    def expert_flops(self, accepted: int) -> int:
        return 4 * self.d * self.d_ff * accepted

    def router_flops(self) -> int:
        cols = (2 if self.noisy else 1) * (self.a + self.a * self.b)
        return 2 * self.T * self.d * cols


# The many-small-experts layer as 16 groups of 64 experts, two of each.
HIER_WORKLOADS = {
    w.name: w
    for w in [
        HierWorkload("hier_16x64_e1024", T=32768, d=512, a=16, b=64, kp=2, ks=2, d_ff=1024,
                     cf=1.5, dtype="bf16", noisy=True),
    ]
}

# Strictly balanced gating (batchwise mask): clean router, m = k*T/E rows per
# expert; the large-expert layer's widths at 64 experts.
BAL_WORKLOADS = {
    w.name: w
    for w in [
        Workload("balanced_top2_e64", T=16384, d=1024, E=64, d_ff=4096, k=2, cf=1.0, mode=TOPK,
                 dtype="bf16", noisy=False),
    ]
}

# The threshold mask (the inference-time form of strictly balanced gating):
# the balanced layer's shapes; k is the bound on a token's picks (the row
# buffers' size), and every expert's threshold is THR_SCALE / E (see
# ``thresholds``).
THR_WORKLOADS = {
    w.name: w
    for w in [
        Workload("threshold_e64", T=16384, d=1024, E=64, d_ff=4096, k=16, cf=1.0, mode=TOPK,
                 dtype="bf16", noisy=False),
    ]
}
THR_SCALE = 4.0


def thresholds(w: Workload) -> np.ndarray:
    """Per-expert thresholds T_i of a threshold workload: the same value
    THR_SCALE / E for every expert, a synthetic stand-in for learned
    thresholds. With this recipe's logits (x ~ N(0, 1), W_g ~ N(0, 1/d)) about
    two experts pass per token, the top-2 regime; since a token's softmax
    gates sum to 1, fewer than E / THR_SCALE (16 here) can pass, so the bound
    k = 16 always holds."""
    return np.full(w.E, THR_SCALE / w.E, np.float32)


_CHUNK = 1 << 24


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def _normal(rng, shape, std: float, as_bf16: bool) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16 if as_bf16 else np.float32)
    s = np.float32(std)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        v = rng.standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            v *= s
        out[lo:hi] = f32_to_bf16_bits(v) if as_bf16 else v
    return out.reshape(shape)


def generate(w: Workload, seed: int = 0, biases: bool = False) -> dict:
    """Draw one input set for ``w``. Returns numpy arrays (bf16 as uint16 bits)
    plus the scalar settings the layer needs."""
    rng = np.random.Generator(np.random.PCG64(seed))
    bf = w.dtype == "bf16"
    x = _normal(rng, (w.T, w.d), 1.0, bf)
    Wg = _normal(rng, (w.d, w.E), w.router_scale / math.sqrt(w.d), False)
    Wn = noise = None
    if w.noisy:
        Wn = _normal(rng, (w.d, w.E), 1.0 / math.sqrt(w.d), False)
        noise = _normal(rng, (w.T, w.E), 1.0, False)
    W1 = _normal(rng, (w.E, w.d, w.d_ff), 1.0 / math.sqrt(w.d), bf)
    b1 = _normal(rng, (w.E, w.d_ff), 0.1, bf) if biases else None
    W2 = _normal(rng, (w.E, w.d_ff, w.d), 1.0 / math.sqrt(w.d_ff), bf)
    b2 = _normal(rng, (w.E, w.d), 0.1, bf) if biases else None
    bias = None
    if w.zipf_bias:
        bias = np.array([1.5 * math.log(1.0 / (e + 1)) for e in range(w.E)], np.float32)
    return dict(x=x, Wg=Wg, Wn=Wn, noise=noise, bias=bias, W1=W1, b1=b1, W2=W2, b2=b2,
                k=w.k, cf=w.cf, min_cap=w.min_cap, mode=1 if w.mode == SWITCH else 0,
                T=w.T, d=w.d, E=w.E, d_ff=w.d_ff)


def generate_dy(w, seed: int = 0) -> np.ndarray:
    """The upstream gradient for the backward: dy ~ N(0, 1) [T, d], drawn
    from its own PCG64 stream (seed + 7919) and rounded to bf16 (uint16 bits)
    for bf16 layers."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    return _normal(rng, (w.T, w.d), 1.0, w.dtype == "bf16")


def generate_hier(w: HierWorkload, seed: int = 0, biases: bool = False) -> dict:
    """Draw one input set for the hierarchical layer ``w`` (same conventions as
    ``generate``)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    bf = w.dtype == "bf16"
    E = w.a * w.b
    x = _normal(rng, (w.T, w.d), 1.0, bf)
    sd = 1.0 / math.sqrt(w.d)
    Wp = _normal(rng, (w.d, w.a), sd, False)
    Wpn = noise_p = None
    if w.noisy:
        Wpn = _normal(rng, (w.d, w.a), sd, False)
        noise_p = _normal(rng, (w.T, w.a), 1.0, False)
    Ws = _normal(rng, (w.d, E), sd, False)
    Wsn = noise_s = None
    if w.noisy:
        Wsn = _normal(rng, (w.d, E), sd, False)
        noise_s = _normal(rng, (w.T, E), 1.0, False)
    W1 = _normal(rng, (E, w.d, w.d_ff), 1.0 / math.sqrt(w.d), bf)
    b1 = _normal(rng, (E, w.d_ff), 0.1, bf) if biases else None
    W2 = _normal(rng, (E, w.d_ff, w.d), 1.0 / math.sqrt(w.d_ff), bf)
    b2 = _normal(rng, (E, w.d), 0.1, bf) if biases else None
    return dict(x=x, Wp=Wp, Wpn=Wpn, noise_p=noise_p, Ws=Ws, Wsn=Wsn, noise_s=noise_s, W1=W1,
                b1=b1, W2=W2, b2=b2, a=w.a, b=w.b, kp=w.kp, ks=w.ks, cf=w.cf,
                min_cap=w.min_cap, T=w.T, d=w.d, d_ff=w.d_ff)
