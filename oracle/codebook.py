"""3-bit Lloyd-Max codebook for N(0,1).

PolyKV abstract: values use "3-bit Lloyd-Max quantization with centroids
tuned to N(0,1)". Lloyd-Max (Lloyd 1957/1982, Max 1960) alternates two
optimality conditions until they hold together:
  * each decision boundary is the midpoint of its two neighbouring centroids;
  * each centroid is the conditional mean of N(0,1) over its cell,
      c_i = (phi(b_{i-1}) - phi(b_i)) / (Phi(b_i) - Phi(b_{i-1})),
    with b_{-1} = -inf and b_{L-1} = +inf.
The iteration runs in float64 and keeps the table symmetric (the density is
even). The fp32 table used for encoding rounds the float64 centroids to fp32
and forms each boundary in fp32 as (c_i + c_{i+1}) * 0.5 from the fp32
centroids, so the middle boundary is exactly 0.
"""
from __future__ import annotations

import math

import numpy as np

SQRT2 = math.sqrt(2.0)
INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)


def _pdf(x: float) -> float:
    return 0.0 if math.isinf(x) else INV_SQRT_2PI * math.exp(-0.5 * x * x)


def _cdf(x: float) -> float:
    return 0.5 * math.erfc(-x / SQRT2)


def lloyd_max_normal(levels: int = 8, tol: float = 1e-13, max_iter: int = 200000):
    """float64 Lloyd-Max centroids and boundaries for N(0,1), ascending."""
    c = [(-(levels - 1) / 2.0 + i) * (4.0 / levels) for i in range(levels)]
    for _ in range(max_iter):
        b = [(c[i] + c[i + 1]) / 2.0 for i in range(levels - 1)]
        edges = [-math.inf] + b + [math.inf]
        new = []
        for i in range(levels):
            lo, hi = edges[i], edges[i + 1]
            new.append((_pdf(lo) - _pdf(hi)) / (_cdf(hi) - _cdf(lo)))
        # the density is symmetric: keep the table exactly antisymmetric
        new = [0.5 * (new[i] - new[levels - 1 - i]) for i in range(levels)]
        delta = max(abs(a - o) for a, o in zip(new, c))
        c = new
        if delta < tol:
            break
    b = [(c[i] + c[i + 1]) / 2.0 for i in range(levels - 1)]
    return np.array(c, dtype=np.float64), np.array(b, dtype=np.float64)


def mse_normal(c: np.ndarray, b: np.ndarray) -> float:
    """E[(X - Q(X))^2] for X ~ N(0,1), closed form per cell [lo, hi]:
    int (x - c)^2 phi = int x^2 phi - 2c int x phi + c^2 int phi, with
    int x phi = phi(lo) - phi(hi) and int x^2 phi = P + lo phi(lo) - hi phi(hi)."""
    edges = [-math.inf] + list(b) + [math.inf]
    total = 0.0
    for i, ci in enumerate(c):
        lo, hi = edges[i], edges[i + 1]
        p = _cdf(hi) - _cdf(lo)
        m1 = _pdf(lo) - _pdf(hi)                       # int x phi
        xlo = 0.0 if math.isinf(lo) else lo * _pdf(lo)
        xhi = 0.0 if math.isinf(hi) else hi * _pdf(hi)
        m2 = p + xlo - xhi                             # int x^2 phi
        total += m2 - 2.0 * ci * m1 + ci * ci * p
    return total


def codebook_f32(levels: int = 8):
    """(centroids fp32[levels], boundaries fp32[levels-1]) used by the encoder."""
    c64, _ = lloyd_max_normal(levels)
    c32 = c64.astype(np.float32)
    b32 = ((c32[:-1] + c32[1:]) * np.float32(0.5)).astype(np.float32)
    return c32, b32
