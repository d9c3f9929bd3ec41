"""Seeded synthetic inputs for fused linear cross-entropy (FLCE).

This module only draws random numbers and rounds them to bf16. It holds none
of the loss arithmetic, so both the CPU oracle and the CUDA path can take
their inputs from it without sharing any of the method.

Every tensor comes from its own counter-based Philox-4x64 stream
(``numpy.random.Philox``) keyed by ``(seed, stream id)``, so a tensor does not
change when another one is resized. Normals are numpy's ziggurat draws in
float32, scaled by the standard deviation in float32 and rounded to bf16 with
round-to-nearest-even (the rounding every GPU library uses for bf16).

Workloads follow the shapes of the pages:

* "Tiny" and "Llama-3-shaped head" shapes and value distributions come from
  the parity and benchmark settings on the Liger-Kernel pages (issue #241,
  parity script; commit 95b01e9, "Performance improvements" table:
  8,192 tokens / hidden 4,096 / vocab 128,256).
* The large-logit case (x, W, b all N(0,1), 8x4096 tokens, H=2048,
  V=128,000) is the parity script of Liger-Kernel issue #241.
* The 256K-vocab case is the memory stress point of DeepSpeed PR #8792
  ("Motivation": 256K vocab, 16K tokens).

Targets are uniform over [0, V) or Zipf(s) (P(k) proportional to
(k+1)^-s, drawn by inverse CDF), with an exact count of rows set to
``ignore_index`` chosen by a seeded permutation.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# Stream ids: one Philox stream per tensor.
_S_X, _S_W, _S_B, _S_Y, _S_IGN, _S_DLOSS, _S_SAMPLE = range(7)

_CHUNK = 1 << 24  # elements drawn per numpy call (bounds host temporaries)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[int(seed), int(stream)]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even).

    Returns the bf16 bit patterns as uint16. Inputs are finite.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_f16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE fp16 (round to nearest, ties to even)."""
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def bits_to_f64(bits: np.ndarray, dtype: str = "bf16") -> np.ndarray:
    """Exact widening of bf16 or fp16 bit patterns to float64."""
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    return bf16_bits_to_f64(bits)


def normal_bf16(seed: int, stream: int, shape, std: float, dtype: str = "bf16") -> np.ndarray:
    """N(0, std^2) samples rounded to bf16 (or fp16); returns uint16 bit patterns."""
    n = int(np.prod(shape))
    g = _rng(seed, stream)
    out = np.empty(n, dtype=np.uint16)
    s = np.float32(std)
    conv = f32_to_f16_bits if dtype == "fp16" else f32_to_bf16_bits
    for i in range(0, n, _CHUNK):
        k = min(_CHUNK, n - i)
        out[i:i + k] = conv(g.standard_normal(k, dtype=np.float32) * s)
    return out.reshape(shape)


def uniform_targets(seed: int, n: int, v: int) -> np.ndarray:
    return _rng(seed, _S_Y).integers(0, v, size=n, dtype=np.int64)


def zipf_targets(seed: int, n: int, v: int, s: float) -> np.ndarray:
    """Class k in [0, v) with probability proportional to (k+1)^-s."""
    w = np.arange(1, v + 1, dtype=np.float64) ** (-float(s))
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = _rng(seed, _S_Y).random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), v - 1).astype(np.int64)


def ignored_rows(seed: int, n: int, count: int) -> np.ndarray:
    """Exactly ``count`` distinct row indices, chosen by a seeded permutation."""
    if count <= 0:
        return np.zeros(0, dtype=np.int64)
    return np.sort(_rng(seed, _S_IGN).permutation(n)[:count]).astype(np.int64)


REDUCTIONS = ("none", "sum", "mean")


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic FLCE problem: shapes, value distributions and options."""
    name: str
    N: int
    H: int
    V: int
    seed: int
    x_std: float = 1.0
    w_std: float = 0.02
    b_std: Optional[float] = None       # None: no bias
    target_dist: str = "uniform"        # "uniform" | "zipf"
    zipf_s: float = 1.1
    ignore_frac: float = 0.0
    ignore_index: int = -100
    label_smoothing: float = 0.0
    lse_square_scale: float = 0.0
    logit_scale: float = 1.0
    reduction: str = "mean"
    dloss: str = "one"                  # "one" | "normal_scalar" | "normal_per_token"
    dtype: str = "bf16"                 # operand type of x, W, b: "bf16" | "fp16"
    dloss_scale: float = 1.0            # multiplies dloss (a loss scale, e.g. 65536)

    @property
    def has_bias(self) -> bool:
        return self.b_std is not None

    @property
    def n_ignored(self) -> int:
        return int(round(self.ignore_frac * self.N))

    def flops_8nhv(self) -> float:
        return 8.0 * self.N * self.H * self.V

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five problem shapes (tiny, medium, Llama-3 head, large logits, 256K vocab).
WORKLOADS = {
    "tiny": Workload("tiny", N=512, H=256, V=4096, seed=1001, ignore_frac=0.05),
    "medium": Workload("medium", N=4096, H=2048, V=32000, seed=1002, b_std=0.02,
                       ignore_frac=0.05, label_smoothing=0.1, lse_square_scale=1e-4),
    "llama3_head": Workload("llama3_head", N=8192, H=4096, V=128256, seed=1003),
    "large_logit": Workload("large_logit", N=32768, H=2048, V=128000, seed=1004,
                            w_std=1.0, b_std=1.0, label_smoothing=0.05,
                            reduction="sum", dloss="normal_scalar"),
    "vocab256k": Workload("vocab256k", N=16384, H=4096, V=262144, seed=1005,
                          target_dist="zipf", zipf_s=1.1, ignore_frac=0.10,
                          logit_scale=0.5, lse_square_scale=1e-4,
                          reduction="none", dloss="normal_per_token"),
}


@dataclasses.dataclass
class Inputs:
    """Host arrays of one workload. bf16 / fp16 tensors are held as uint16 bit
    patterns (the workload's dtype says which)."""
    wl: Workload
    x: np.ndarray            # uint16 [N, H]
    W: np.ndarray            # uint16 [V, H]
    b: Optional[np.ndarray]  # uint16 [V] or None
    y: np.ndarray            # int64 [N]
    dloss: np.ndarray        # float32 [1] (mean/sum) or [N] (none)


def make_inputs(wl: Workload) -> Inputs:
    x = normal_bf16(wl.seed, _S_X, (wl.N, wl.H), wl.x_std, wl.dtype)
    W = normal_bf16(wl.seed, _S_W, (wl.V, wl.H), wl.w_std, wl.dtype)
    b = normal_bf16(wl.seed, _S_B, (wl.V,), wl.b_std, wl.dtype) if wl.has_bias else None
    if wl.target_dist == "uniform":
        y = uniform_targets(wl.seed, wl.N, wl.V)
    elif wl.target_dist == "zipf":
        y = zipf_targets(wl.seed, wl.N, wl.V, wl.zipf_s)
    else:
        raise ValueError(wl.target_dist)
    y[ignored_rows(wl.seed, wl.N, wl.n_ignored)] = wl.ignore_index
    g = _rng(wl.seed, _S_DLOSS)
    if wl.dloss == "one":
        dloss = np.ones(1, dtype=np.float32)
    elif wl.dloss == "normal_scalar":
        dloss = g.standard_normal(1, dtype=np.float32)
    elif wl.dloss == "normal_per_token":
        dloss = g.standard_normal(wl.N, dtype=np.float32)
    else:
        raise ValueError(wl.dloss)
    if wl.reduction != "none" and dloss.size != 1:
        raise ValueError("a reduced loss takes a scalar upstream gradient")
    if wl.dloss_scale != 1.0:
        dloss = (dloss * np.float32(wl.dloss_scale)).astype(np.float32)
    return Inputs(wl, x, W, b, y, dloss)


def sample_indices(seed: int, n: int, count: int, must_include=()) -> np.ndarray:
    """Seeded sorted sample of ``count`` distinct indices in [0, n), forced to
    contain ``must_include`` (used to sample rows for large-size parity)."""
    must = np.unique(np.asarray(list(must_include), dtype=np.int64))
    must = must[(must >= 0) & (must < n)]
    count = min(count, n)
    perm = _rng(seed, _S_SAMPLE).permutation(n)
    rest = perm[~np.isin(perm, must)][: max(0, count - must.size)]
    return np.sort(np.concatenate([must, rest]).astype(np.int64))
