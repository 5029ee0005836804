"""Seeded synthetic logit rows for the top-k / top-p filter tests: random
values with ties, signed zeros, masked (-inf) ids and flat stretches.  Input
generation only; no filtering arithmetic here."""
from __future__ import annotations

import numpy as np

import synth


def rows(seed: int, n: int, V: int, dtype: str, sigma: float = 3.0) -> np.ndarray:
    """[n, V] logits as float32 or bf16 bit patterns (uint16)."""
    rng = np.random.default_rng(seed)
    z = (sigma * rng.standard_normal((n, V)) - 1.1 * np.log1p(np.arange(V))).astype(np.float32)
    for r in range(n):
        kind = r % 4
        if kind == 1:       # ties: values on a coarse grid
            z[r] = np.round(z[r] * 2.0) / 2.0
        elif kind == 2:     # masked ids and signed zeros
            z[r][rng.random(V) < 0.3] = -np.inf
            zs = rng.random(V) < 0.05
            z[r][zs] = np.where(rng.random(zs.sum()) < 0.5, 0.0, -0.0)
            if not np.isfinite(z[r]).any():
                z[r][0] = 0.0
        elif kind == 3:     # a flat stretch of equal values at the top
            z[r][: max(1, V // 3)] = z[r].max() + 1.0
    if dtype == "bf16":
        return synth.f32_to_bf16(z)
    return z
