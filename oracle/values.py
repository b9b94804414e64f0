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
  * packing (3 bits per code, no padding): the pool keeps codes in groups of
    32 consecutive tokens of one (layer, kv head); for each coordinate j the
    group's 32 codes form one little-endian 96-bit (12-byte) string, token k
    of the group at bits 3k..3k+2, and the d strings of a group follow in
    coordinate order (12*d bytes per 32 tokens = 3d/8 bytes per token);
  * the stored norm is fp16 (round to nearest even); the codes use the
    unrounded fp32 norm.
Dequantized value: v_hat = H_n((n16 / sqrt(d)) * C[code]) = (n16 / d) * H C[code].
"""
from __future__ import annotations

import numpy as np


def butterfly(a, b):
    """One Walsh-Hadamard butterfly: (a, b) -> (a + b, a - b), a the lower index."""
    return a + b, a - b


def fwht_f32_pinned(v: np.ndarray) -> np.ndarray:
    """Unnormalized Sylvester FWHT along the last axis in fp32, strides 1, 2, 4, ..."""
    y = np.array(v, dtype=np.float32, copy=True)
    d = y.shape[-1]
    lead = y.shape[:-1]
    h = 1
    while h < d:
        y = y.reshape(lead + (d // (2 * h), 2, h))
        y = np.stack(butterfly(y[..., 0, :], y[..., 1, :]), axis=-2).astype(np.float32)
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
        y = np.stack(butterfly(y[..., 0, :], y[..., 1, :]), axis=-2)
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


GROUP = 32  # tokens per packed code group


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 codes [..., T, d] (T a multiple of 32) -> packed bytes [..., T/32, d, 12]:
    string (group, j) holds token k of the group at bits 3k..3k+2 (little endian)."""
    c = np.asarray(codes, dtype=np.uint8)
    T, d = c.shape[-2], c.shape[-1]
    assert T % GROUP == 0, "pack_codes takes whole 32-token groups"
    g = c.reshape(c.shape[:-2] + (T // GROUP, GROUP, d))
    g = np.swapaxes(g, -1, -2)                                   # [..., G, d, 32 tokens]
    bits = np.stack([(g >> b) & 1 for b in range(3)], axis=-1)   # [..., G, d, 32, 3]: bit 3k+b
    bits = bits.reshape(bits.shape[:-2] + (3 * GROUP,)).astype(np.uint8)
    return np.packbits(bits, axis=-1, bitorder="little")         # [..., G, d, 12]


def unpack_codes(packed: np.ndarray, d: int) -> np.ndarray:
    """packed bytes [..., G, d, 12] -> uint8 codes [..., 32*G, d]."""
    p = np.asarray(packed, dtype=np.uint8)
    assert p.shape[-2] == d and p.shape[-1] == 3 * GROUP // 8
    bits = np.unpackbits(p, axis=-1, bitorder="little").reshape(p.shape[:-1] + (GROUP, 3))
    codes = (bits[..., 0] | (bits[..., 1] << 1) | (bits[..., 2] << 2)).astype(np.uint8)   # [..., G, d, 32]
    codes = np.swapaxes(codes, -1, -2)                                                      # [..., G, 32, d]
    return codes.reshape(codes.shape[:-3] + (codes.shape[-3] * GROUP, d))


def dequantize_values(codes: np.ndarray, norm16: np.ndarray, centroids_f32: np.ndarray) -> np.ndarray:
    """float64 v_hat = (n16 / d) * H C[code]."""
    d = codes.shape[-1]
    cvals = centroids_f32.astype(np.float64)[codes.astype(np.int64)]
    return fwht_f64(cvals) * (norm16.astype(np.float64) / d)[..., None]
