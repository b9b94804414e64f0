"""q8_0 key quantization.

PolyKV abstract: "Keys are quantized at int8 (q8_0) to preserve softmax
stability". q8_0 is the GGML block format: blocks of 32 consecutive
elements, one fp16 scale per block, int8 codes. Readings taken here:
  * blocks run along head_dim inside each (layer, kv head, token) key vector;
  * amax is taken in fp32 over the block; scale s16 = fp16_rne(fp32(amax / 127));
  * each code is round-half-away-from-zero of the correctly rounded fp32
    quotient x / s16 (dividing by the STORED scale, so |x - q*s16| <= s16/2),
    clamped to [-127, 127];
  * a block whose s16 is 0 (or not finite) gets all-zero codes.
Dequantized key: k_hat_j = s16[block(j)] * q_j.
"""
from __future__ import annotations

import numpy as np

BLOCK = 32


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(bits) if dtype == "bf16" else f16_bits_to_f32(bits)


def round_half_away(r64: np.ndarray) -> np.ndarray:
    """Nearest integer, ties away from zero (q8_0's rounding), exact in float64."""
    return np.sign(r64) * np.floor(np.abs(r64) + 0.5)


def quantize_q8_0(x: np.ndarray):
    """x: fp32 [..., d] (d a multiple of 32). Returns (codes int8 [..., d], scales fp16 [..., d/32])."""
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    assert d % BLOCK == 0
    xb = x.reshape(x.shape[:-1] + (d // BLOCK, BLOCK))
    amax = np.max(np.abs(xb), axis=-1)                          # fp32, exact
    with np.errstate(over="ignore"):
        s16 = (amax / np.float32(127.0)).astype(np.float16)     # fp32 divide, then fp16 RNE
    sf = s16.astype(np.float32)
    usable = (sf > 0) & np.isfinite(sf)
    safe = np.where(usable, sf, np.float32(1.0))[..., None]
    r = (xb / safe).astype(np.float32)                          # correctly rounded fp32 quotient
    q = np.clip(round_half_away(r.astype(np.float64)), -127, 127)
    q = np.where(usable[..., None], q, 0.0)
    return q.astype(np.int8).reshape(x.shape), s16


def dequantize_q8_0(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """float64 k_hat from int8 codes [..., d] and fp16 scales [..., d/32]."""
    d = codes.shape[-1]
    s = np.repeat(scales.astype(np.float64), BLOCK, axis=-1)
    assert s.shape[-1] == d
    return codes.astype(np.float64) * s
