"""Seeded synthetic inputs for the ternary-weight linear layer.

This module only draws random numbers and rounds them to the storage types the
layer consumes (int8 ternary weights, fp16 group scales, bf16 activations).  It
holds none of the layer's arithmetic (no packing, no quantisation, no
products), so the CPU oracle and the CUDA path can both take their inputs from
it without sharing any of the method.

The shapes and distributions stand in for the pages' model weights and
perplexity corpus, which are not available: 27B-like projections (fused
gate+up 5120x34816, down 17408x5120, attention-like 5120x6144 and 6144x5120),
ternary weights with a chosen zero fraction, one fp16 scale per 128 weights,
bf16 N(0,1) activations with 1% of channels scaled x20 as outliers.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# Projection shapes (K inputs, N outputs).
SHAPES = {
    "tiny": (512, 1024),
    "gu": (5120, 2 * 17408),   # fused gate+up
    "dn": (17408, 5120),       # down
    "ai": (5120, 6144),        # attention-like in
    "ao": (6144, 5120),        # attention-like out
}

GROUP = 128

# Stream tags so that each tensor of a case draws from its own stream.
_TAG_W, _TAG_S, _TAG_X, _TAG_OUT = 1, 2, 3, 4


def _rng(seed: int, tag: int, extra: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(tag), int(extra)])


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns with round-to-nearest-even (finite inputs)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def ternary_weights(N: int, K: int, p_zero: float, seed: int, extra: int = 0) -> np.ndarray:
    """int8 [N, K] with P(0) = p_zero and P(+1) = P(-1) = (1 - p_zero) / 2.

    p_zero must be a multiple of 1/30 (covers 1/3, 0.2, 0.4, 0.6)."""
    z = int(round(p_zero * 30))
    assert abs(z / 30 - p_zero) < 1e-9 and 0 <= z <= 30 and (30 - z) % 2 == 0
    r = _rng(seed, _TAG_W, extra).integers(0, 30, size=(N, K), dtype=np.uint8)
    half = (30 - z) // 2
    w = np.zeros((N, K), dtype=np.int8)
    w[(r >= z) & (r < z + half)] = 1
    w[r >= z + half] = -1
    return w


def scales_uniform(N: int, K: int, lo: float, hi: float, seed: int, extra: int = 0) -> np.ndarray:
    """fp16 [N, K/128], uniform in [lo, hi] rounded to fp16."""
    g = K // GROUP
    return _rng(seed, _TAG_S, extra).uniform(lo, hi, size=(N, g)).astype(np.float16)


def scales_lognormal(N: int, K: int, mu: float, sigma: float, seed: int, extra: int = 0) -> np.ndarray:
    """fp16 [N, K/128], exp(N(mu, sigma^2)) rounded to fp16."""
    g = K // GROUP
    return np.exp(_rng(seed, _TAG_S, extra).normal(mu, sigma, size=(N, g))).astype(np.float16)


def activations(T: int, K: int, seed: int, outlier_frac: float = 0.0,
                outlier_gain: float = 20.0, extra: int = 0) -> np.ndarray:
    """bf16 bit patterns [T, K]: N(0,1) in fp32, a fixed seeded set of
    round(outlier_frac*K) channels (the same for every token) multiplied by
    outlier_gain in fp32, then rounded to bf16 (RNE)."""
    rng = _rng(seed, _TAG_X, extra)
    x = rng.standard_normal(size=(T, K), dtype=np.float32)
    n_out = int(round(outlier_frac * K))
    if n_out:
        ch = _rng(seed, _TAG_OUT, extra).choice(K, size=n_out, replace=False)
        x[:, ch] *= np.float32(outlier_gain)
    return f32_to_bf16_bits(x)


@dataclass
class Case:
    """One projection at one token count, as host arrays."""
    name: str
    T: int
    K: int
    N: int
    W: np.ndarray        # int8 [N, K]
    scales: np.ndarray   # fp16 [N, K/128]
    x: np.ndarray        # uint16 bf16 bits [T, K]


def case(name: str, T: int, *, seed: int = 0, p_zero: float = 0.4, scale_kind: str = "lognormal",
         outliers: bool = True, K: int | None = None, N: int | None = None, extra: int = 0) -> Case:
    """A projection case.  ``name`` picks the shape from SHAPES unless K, N are given.

    scale_kind: "lognormal" (mu=-3.5, sigma=0.3) or "uniform" ([0.01, 0.05]).
    outliers: 1% of channels x20."""
    if K is None or N is None:
        K, N = SHAPES[name]
    W = ternary_weights(N, K, p_zero, seed, extra)
    if scale_kind == "uniform":
        s = scales_uniform(N, K, 0.01, 0.05, seed, extra)
    else:
        s = scales_lognormal(N, K, -3.5, 0.3, seed, extra)
    x = activations(T, K, seed, 0.01 if outliers else 0.0, extra=extra)
    return Case(name, T, K, N, W, s, x)


# The five workload families.
def config_tiny() -> Case:
    """Tiny: K=512, N=1024, T=1, uniform ternary, U[0.01,0.05] scales, plain N(0,1) x, seed 0."""
    return case("tiny", 1, seed=0, p_zero=1.0 / 3.0, scale_kind="uniform", outliers=False)


def config_decode(proj: str) -> Case:
    """Decode GEMV at T=1 for 'gu' or 'dn': P(0)=0.4, lognormal scales, 1% outliers."""
    return case(proj, 1, seed=0, p_zero=0.4, scale_kind="lognormal", outliers=True)


def config_verify(proj: str, T: int) -> Case:
    """Speculative-verify band, T in 2..16: independent plain N(0,1) rows."""
    return case(proj, T, seed=0, p_zero=0.4, scale_kind="lognormal", outliers=False)


def config_prefill(proj: str, T: int) -> Case:
    """Prefill s8 band, T >= 17, on gu/dn/ai/ao: activations with outliers."""
    return case(proj, T, seed=0, p_zero=0.4, scale_kind="lognormal", outliers=True)


VERIFY_T = (2, 3, 4, 8, 9, 12, 16)
PREFILL_T = (17, 508, 2048)
STACK_LAYERS = 64
STACK_PROJ = ("gu", "dn", "ai", "ao")
STACK_P_ZERO = (0.2, 0.4, 0.6)
STACK_SEEDS = (1, 2, 3)
