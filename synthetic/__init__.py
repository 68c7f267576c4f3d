"""Seeded synthetic inputs for the quantized decode GEMV.

This module only draws random numbers.  It holds none of the method's
arithmetic: no quantization, no dequantization, no dot products, no knowledge
of any block layout.  The CPU oracle, the tests and the benchmark all take
their inputs from here, so every side sees the same fp32 data for a seed.

Workload recipe (stand-in for Llama-7B / 8B-class decode, where no real
checkpoint is used):
  * weights  W[M][K]  fp32 ~ N(0, 0.02), row-major;
  * activations x[ncols][K] fp32 ~ N(0, 1); optionally a fraction of each
    column's entries (1 % in the outlier workload) multiplied by 20, the
    positions chosen by a seeded permutation;
  * MoE routing ids[n_tokens][top_k] int32, for each token top_k distinct
    experts drawn uniformly without replacement.

Two generators are provided: numpy's PCG64 on the host (bit-reproducible
across machines; used for everything the oracle has to see) and torch's
device Philox generator (used only for benchmark-sized weights, which the
oracle never checks element by element).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "host_rng",
    "normal_f32",
    "weights_f32",
    "activations_f32",
    "moe_ids",
    "uniform_u8",
    "uniform_int",
    "device_normal_f32",
]


def host_rng(seed: int) -> np.random.Generator:
    """numpy PCG64 generator for ``seed``."""
    return np.random.Generator(np.random.PCG64(int(seed)))


def normal_f32(seed: int, shape, sigma: float = 1.0) -> np.ndarray:
    """fp32 samples of N(0, sigma^2) with the given shape."""
    g = host_rng(seed)
    a = g.standard_normal(shape, dtype=np.float32)
    if sigma != 1.0:
        a *= np.float32(sigma)
    return a


def weights_f32(seed: int, M: int, K: int, sigma: float = 0.02) -> np.ndarray:
    """Row-major fp32 weight matrix W[M][K] ~ N(0, sigma^2)."""
    return normal_f32(seed, (M, K), sigma)


def activations_f32(seed: int, ncols: int, K: int, outlier_frac: float = 0.0,
                    outlier_scale: float = 20.0) -> np.ndarray:
    """fp32 activation columns x[ncols][K] ~ N(0, 1).

    With ``outlier_frac`` > 0, round(outlier_frac * K) positions of every
    column (a seeded permutation prefix, independent per column) are
    multiplied by ``outlier_scale``.
    """
    g = host_rng(seed)
    x = g.standard_normal((ncols, K), dtype=np.float32)
    n_out = int(round(outlier_frac * K))
    if n_out > 0:
        for c in range(ncols):
            idx = g.permutation(K)[:n_out]
            x[c, idx] *= np.float32(outlier_scale)
    return x


def moe_ids(seed: int, n_tokens: int, top_k: int, n_expert: int) -> np.ndarray:
    """int32 ids[n_tokens][top_k]: per token, top_k distinct experts drawn
    uniformly without replacement."""
    if top_k > n_expert:
        raise ValueError("top_k > n_expert")
    g = host_rng(seed)
    ids = np.empty((n_tokens, top_k), dtype=np.int32)
    for t in range(n_tokens):
        ids[t] = g.choice(n_expert, size=top_k, replace=False)
    return ids


def uniform_u8(seed: int, n: int) -> np.ndarray:
    """n uniformly random bytes."""
    return host_rng(seed).integers(0, 256, size=n, dtype=np.uint8)


def uniform_int(seed: int, shape, lo: int, hi: int) -> np.ndarray:
    """int64 samples uniform on [lo, hi] inclusive."""
    return host_rng(seed).integers(lo, hi + 1, size=shape, dtype=np.int64)


def device_normal_f32(seed: int, shape, sigma: float, device):
    """fp32 N(0, sigma^2) drawn on a CUDA device by torch's Philox generator.

    Used for benchmark-sized weight sets (gigabytes) that are too slow to draw
    on the host.  Reproducible for a given torch build and device type.
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if sigma != 1.0:
        t.mul_(sigma)
    return t
