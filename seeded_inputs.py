"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module draws random numbers and rounds them to bf16; it holds none of the
attention arithmetic.  Both the CUDA path and the oracle receive the very same
bf16 tensors, and the oracle widens them to float64 itself.

Recipe (one generator per workload, drawn in the order Q, K, V, dO):

    rng = numpy.random.default_rng(seed)
    X   = rng.standard_normal((B, H, N, d), dtype=float32)   for X in Q, K, V, dO
    X   = torch.from_numpy(X).to(torch.bfloat16)              # round-to-nearest-even

The "large-logit" variant multiplies the bf16 Q and K by 4 afterwards (a power
of two, so the product is exact in bf16).  Rows of the row sample used at long
context come from a second generator seeded with ``seed + 1000``.

The shapes below are the workloads of exact tiled attention at head size
32/64/128 and sequence lengths 256 to 32768.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: tuple  # which masking modes the workload runs
    seed: int
    qk_mult: float = 1.0  # multiplier on Q and K (large-logit stress)
    sample_rows: int = 0  # >0: the oracle checks this many rows per head

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def fwd_flops(self, causal: bool) -> float:
        """4 N^2 d per head for the forward, halved under the causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f * 0.5 if causal else f

    def bwd_flops(self, causal: bool) -> float:
        """10 N^2 d per head for the backward, halved under the causal mask."""
        f = 10.0 * self.B * self.H * self.N * self.N * self.d
        return f * 0.5 if causal else f


WORKLOADS = {
    # tiny exactness case: fp64 oracle runs in well under a second
    "tiny_1x1x256x32": Workload("tiny_1x1x256x32", 1, 1, 256, 32, (False, True), seed=0),
    # small training shape
    "small_4x8x1024x64": Workload("small_4x8x1024x64", 4, 8, 1024, 64, (True,), seed=1),
    # mid shape, both mask modes
    "mid_2x16x4096x128": Workload("mid_2x16x4096x128", 2, 16, 4096, 128, (False, True), seed=2),
    # long context, unit-variance and large-logit (Q,K x4) variants
    "long_1x32x8192x128": Workload("long_1x32x8192x128", 1, 32, 8192, 128, (True,), seed=3),
    "long_1x32x8192x128_qk4": Workload("long_1x32x8192x128_qk4", 1, 32, 8192, 128, (True,), seed=3,
                                       qk_mult=4.0),
    # very long context: only O and L are stored; the oracle checks sampled rows
    "vlong_1x32x32768x128": Workload("vlong_1x32x32768x128", 1, 32, 32768, 128, (True,), seed=4,
                                     sample_rows=256),
}


def make_qkvdo(B: int, H: int, N: int, d: int, seed: int, qk_mult: float = 1.0):
    """Return (Q, K, V, dO) as contiguous bf16 CPU tensors of shape [B, H, N, d]."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(4):
        x = rng.standard_normal((B, H, N, d), dtype=np.float32)
        out.append(torch.from_numpy(x).to(torch.bfloat16))
    if qk_mult != 1.0:
        out[0] = (out[0] * qk_mult).contiguous()
        out[1] = (out[1] * qk_mult).contiguous()
    return tuple(out)


def make_workload(w: Workload):
    return make_qkvdo(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)


def sample_rows(w: Workload, n_rows: int | None = None) -> np.ndarray:
    """Sorted row indices (per head, the same for every head) for sampled checks."""
    n = n_rows or w.sample_rows or w.N
    if n >= w.N:
        return np.arange(w.N)
    rng = np.random.default_rng(w.seed + 1000)
    rows = rng.choice(w.N, size=n, replace=False)
    # always include the first and last rows: the causal extremes
    rows[0], rows[1] = 0, w.N - 1
    return np.unique(rows)


def to_f64(t: torch.Tensor) -> np.ndarray:
    """bf16 (or any float) tensor -> float64 numpy array (exact widening)."""
    return t.detach().to("cpu").to(torch.float64).numpy()
