"""Seeded inputs for the sharded (ZeRO-1) data-parallel step tests.

Each rank holds its own full gradient.  Its values are small integers times a power
of two (FP32: k * 2^-20 with |k| < 2^20; BF16: k * 2^-12 with |k| <= 15), so the sum
over up to four ranks is exact in the storage type whatever order a collective adds
them in, and the reduced gradient the oracle takes is that exact sum.  Nothing here
computes any part of the optimizer.
"""

from __future__ import annotations

import numpy as np

SEED = 77


def rank_gradient(n: int, padded: int, rank: int, call: int, dtype: str,
                  inf_at: int | None = None) -> np.ndarray:
    """Rank's stored gradient for 1-based ``call``, ``padded`` elements (zero past n):
    float32 values, or uint16 BF16 bit patterns."""
    rng = np.random.default_rng([SEED, rank, call])
    if dtype == "f32":
        x = (rng.integers(-(1 << 19), 1 << 19, n) * 2.0 ** -20).astype(np.float32)
    else:
        x = (rng.integers(-15, 16, n) * 2.0 ** -12).astype(np.float32)
    if inf_at is not None:
        x[inf_at] = np.float32(np.inf)
    out = np.zeros(padded, np.float32)
    out[:n] = x
    if dtype == "f32":
        return out
    return (out.view(np.uint32) >> 16).astype(np.uint16)  # exact: values fit in BF16


def reduced_gradient(n: int, world: int, call: int, dtype: str,
                     inf: tuple[int, int, int] | None = None) -> np.ndarray:
    """The sum over ranks of the first n elements (exact), in the storage type.
    ``inf`` = (call, rank, index) plants +Inf in that rank's gradient."""
    total = np.zeros(n, np.float64)
    for r in range(world):
        at = inf[2] if inf is not None and inf[0] == call and inf[1] == r else None
        g = rank_gradient(n, n, r, call, dtype, at)
        total += g.astype(np.float64) if dtype == "f32" else \
            (g.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    x = total.astype(np.float32)
    if dtype == "f32":
        return x
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def params(n: int) -> np.ndarray:
    rng = np.random.default_rng([SEED, 1000])
    return (rng.standard_normal(n) * 0.02).astype(np.float32)
