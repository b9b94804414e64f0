"""Memory accounting of the compressed pool.

PolyKV abstract: "a stable 2.91x compression ratio across all
configurations" and, for Llama-3-8B with 15 agents sharing a 4K-token
context, KV memory "from 19.8 GB to 0.45 GB -- a 97.7% reduction".
Nominal accounting counts 8 bits per key element and 3 bits per value
element against 16 + 16 for an fp16 cache and ignores the per-block scale
and per-vector norm: (16 + 16) / (8 + 3) = 2.909. The exact accounting of
this pool format adds one fp16 scale per 32 key elements and one fp16 norm
per value vector.
"""
from __future__ import annotations


def nominal_ratio() -> float:
    return (16.0 + 16.0) / (8.0 + 3.0)


def exact_bits_per_element(head_dim: int) -> tuple[float, float]:
    """(key bits, value bits) per element including scale and norm overheads."""
    return 8.0 + 16.0 / 32.0, 3.0 + 16.0 / head_dim


def exact_ratio(head_dim: int) -> float:
    kb, vb = exact_bits_per_element(head_dim)
    return 32.0 / (kb + vb)


def shared_pool_reduction(n_agents: int, ratio: float) -> float:
    """Fraction of memory saved by one compressed pool vs n_agents fp16 caches."""
    return 1.0 - 1.0 / (n_agents * ratio)


def pool_bytes(n_layers, n_kv_heads, n_tokens, head_dim) -> int:
    per = head_dim + 2 * (head_dim // 32) + 3 * head_dim // 8 + 2
    return n_layers * n_kv_heads * n_tokens * per


def fp16_cache_bytes(n_layers, n_kv_heads, n_tokens, head_dim) -> int:
    return n_layers * n_kv_heads * n_tokens * head_dim * 2 * 2
