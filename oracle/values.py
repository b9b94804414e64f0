"""Value compression: FWHT rotation, norm scaling, 3-bit Lloyd-Max codes.

PolyKV abstract: values are compressed with "TurboQuant MSE -- a Fast
Walsh-Hadamard Transform (FWHT) rotation followed by 3-bit Lloyd-Max
quantization with centroids tuned to N(0,1)". The rotation is the
normalized Hadamard transform H_n = H / sqrt(d) over head_dim; the rotated
vector is scaled by sqrt(d) / ||v|| so its coordinates are about N(0,1), and
||v|| is stored with the codes. Since (sqrt(d)/||v||) * (H v / sqrt(d)) =
H v / ||v||, the encoder forms u = (H v) / ||v|| with the UNnormalized
Sylvester transform H and one correctly rounded division.

Readings taken (the abstract is silent on them):
  * natural (Sylvester) Hadamard order, no random sign flips;
  * fp32 arithmetic in a fixed order, shared with the GPU encoder:
      - ||v||^2: per group of 8 consecutive coordinates a left-to-right sum
        of rounded squares (no fused multiply-add), then a balanced pairwise
        tree over the d/8 group sums; ||v|| = correctly rounded sqrt;
      - butterflies at strides h = 1, 2, 4, ..., d/2, each pair
        (a, b) -> (a + b, a - b) with a the lower index;
      - u_j = y_j / ||v|| correctly rounded; u = 0 when ||v|| = 0;
  * code_j = #{i : u_j >= b_i} over the 7 fp32 boundaries (ties go up);
  * 8 codes per 3 bytes: coordinate 8g+i sits at bits 3i..3i+2 of a
    little-endian 24-bit word (d=128 -> 48 bytes, d=64 -> 24 bytes);
  * the stored norm is fp16 (round to nearest even); the codes use the
    unrounded fp32 norm.
Dequantized value: v_hat = H_n((n16 / sqrt(d)) * C[code]) = (n16 / d) * H C[code].
"""
from __future__ import annotations

import numpy as np


def fwht_f32_pinned(v: np.ndarray) -> np.ndarray:
    """Unnormalized Sylvester FWHT along the last axis in fp32, strides 1, 2, 4, ..."""
    y = np.array(v, dtype=np.float32, copy=True)
    d = y.shape[-1]
    lead = y.shape[:-1]
    h = 1
    while h < d:
        y = y.reshape(lead + (d // (2 * h), 2, h))
        a = y[..., 0, :]
        b = y[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).astype(np.float32)
        h *= 2
    return y.reshape(lead + (d,))


def fwht_f64(v: np.ndarray) -> np.ndarray:
    """Unnormalized Sylvester FWHT along the last axis in float64."""
    y = np.array(v, dtype=np.float64, copy=True)
    d = y.shape[-1]
    lead = y.shape[:-1]
    h = 1
    while h < d:
        y = y.reshape(lead + (d // (2 * h), 2, h))
        a = y[..., 0, :]
        b = y[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2)
        h *= 2
    return y.reshape(lead + (d,))


def sumsq_f32_pinned(v: np.ndarray) -> np.ndarray:
    """||v||^2 in fp32 in the fixed order described in the module docstring."""
    v = np.asarray(v, dtype=np.float32)
    d = v.shape[-1]
    sq = (v * v).astype(np.float32).reshape(v.shape[:-1] + (d // 8, 8))
    acc = sq[..., 0].copy()
    for i in range(1, 8):
        acc = (acc + sq[..., i]).astype(np.float32)
    while acc.shape[-1] > 1:
        acc = (acc[..., 0::2] + acc[..., 1::2]).astype(np.float32)
    return acc[..., 0]


def rotate_normalize(v: np.ndarray):
    """Returns (u fp32 [..., d], n fp32 [...]): u = (H v) / ||v||."""
    n = np.sqrt(sumsq_f32_pinned(v)).astype(np.float32)
    y = fwht_f32_pinned(v)
    safe = np.where(n > 0, n, np.float32(1.0))[..., None]
    u = np.where((n > 0)[..., None], (y / safe).astype(np.float32), np.float32(0.0))
    return u.astype(np.float32), n


def quantize_u(u: np.ndarray, boundaries_f32: np.ndarray) -> np.ndarray:
    """code = number of boundaries b_i with u >= b_i (uint8 in 0..7)."""
    return np.sum(u[..., None] >= boundaries_f32.astype(np.float32), axis=-1).astype(np.uint8)


def encode_values(v: np.ndarray, boundaries_f32: np.ndarray):
    """v fp32 [..., d] -> (codes uint8 [..., d], norm fp16 [...], u fp32 [..., d])."""
    u, n = rotate_normalize(v)
    codes = quantize_u(u, boundaries_f32)
    return codes, n.astype(np.float16), u


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 codes [..., d] -> packed bytes [..., 3d/8]."""
    c = np.asarray(codes, dtype=np.uint32)
    d = c.shape[-1]
    g = c.reshape(c.shape[:-1] + (d // 8, 8))
    w = np.zeros(g.shape[:-1], dtype=np.uint32)
    for i in range(8):
        w |= g[..., i] << np.uint32(3 * i)
    out = np.stack([w & 0xFF, (w >> 8) & 0xFF, (w >> 16) & 0xFF], axis=-1).astype(np.uint8)
    return out.reshape(c.shape[:-1] + (3 * d // 8,))


def unpack_codes(packed: np.ndarray, d: int) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint32).reshape(packed.shape[:-1] + (d // 8, 3))
    w = p[..., 0] | (p[..., 1] << np.uint32(8)) | (p[..., 2] << np.uint32(16))
    out = np.stack([(w >> np.uint32(3 * i)) & 7 for i in range(8)], axis=-1).astype(np.uint8)
    return out.reshape(packed.shape[:-1] + (d,))


def dequantize_values(codes: np.ndarray, norm16: np.ndarray, centroids_f32: np.ndarray) -> np.ndarray:
    """float64 v_hat = (n16 / d) * H C[code]."""
    d = codes.shape[-1]
    cvals = centroids_f32.astype(np.float64)[codes.astype(np.int64)]
    return fwht_f64(cvals) * (norm16.astype(np.float64) / d)[..., None]
