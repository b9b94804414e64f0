"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module only draws random numbers and casts them to the storage dtypes
(fp16 / bf16 bit patterns, round-to-nearest-even). It contains none of the
PolyKV arithmetic: no quantization, no rotation, no attention.

Workload shapes follow the models and contexts named in the PolyKV abstract
("PolyKV: A Shared Asymmetrically-Compressed KV Cache Pool for Multi-Agent
LLM Inference", abstract: SmolLM2-1.7B-Instruct and Llama-3-8B-Instruct,
600-7,194-token contexts, up to 15 agents). Trained weights and evaluation
text are not available, so tensors are drawn from the stated distributions:

* K = N(0,1) * s_c with a per-(layer, kv head, channel) outlier scale
  s_c = exp(N(0,1)), fixed across tokens (post-RoPE keys with channel
  outliers);
* V = N(0,1);
* q = N(0,1) / 8.

One numpy PCG64 stream per tensor, spawned from SeedSequence(seed).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F16 = "f16"
BF16 = "bf16"


@dataclass(frozen=True)
class Workload:
    name: str
    n_layers: int
    n_kv_heads: int
    n_q_heads: int
    head_dim: int
    n_ctx: int
    n_agents: int
    dtype: str
    suffix_len: int = 0
    note: str = ""

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def describe(self) -> dict:
        d = {
            "workload": self.name,
            "n_layers": self.n_layers,
            "n_kv_heads": self.n_kv_heads,
            "n_q_heads": self.n_q_heads,
            "head_dim": self.head_dim,
            "n_ctx": self.n_ctx,
            "n_agents": self.n_agents,
            "dtype": self.dtype,
        }
        if self.suffix_len:
            d["suffix_len"] = self.suffix_len
        return d


WORKLOADS = {
    # SmolLM2-1.7B shape, a single layer, one agent (small parity case).
    "smollm2_1layer_600": Workload("smollm2_1layer_600", 1, 32, 32, 64, 600, 1, F16),
    # SmolLM2-1.7B shape, full stack, 1851-token shared context, 5 agents.
    "smollm2_24l_1851_a5": Workload("smollm2_24l_1851_a5", 24, 32, 32, 64, 1851, 5, F16),
    # Llama-3-8B shape, 4096-token shared context, 15 agents (GQA group 4).
    "llama3_8b_4096_a15": Workload("llama3_8b_4096_a15", 32, 8, 32, 128, 4096, 15, BF16),
    # Llama-3-8B shape, 7194-token pool plus a private 256-token bf16 suffix per agent.
    "llama3_8b_7194_a15_sfx256": Workload("llama3_8b_7194_a15_sfx256", 32, 8, 32, 128, 7194, 15, BF16,
                                          suffix_len=256),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> fp16 bit patterns (numpy's cast is round to nearest even)."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x) if dtype == BF16 else f32_to_f16_bits(x)


def _streams(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def gen_kv(n_layers, n_kv_heads, n_tokens, head_dim, dtype, seed=0):
    """K, V as uint16 bit patterns, shape [n_layers][n_kv_heads][n_tokens][head_dim]."""
    g_scale, g_k, g_v, _ = _streams(seed, 4)
    chan = np.exp(g_scale.standard_normal((n_layers, n_kv_heads, 1, head_dim), dtype=np.float32))
    k = g_k.standard_normal((n_layers, n_kv_heads, n_tokens, head_dim), dtype=np.float32)
    k *= chan
    kb = to_bits(k, dtype)
    del k
    v = g_v.standard_normal((n_layers, n_kv_heads, n_tokens, head_dim), dtype=np.float32)
    vb = to_bits(v, dtype)
    return kb, vb


def gen_q(n_layers, n_agents, n_q_heads, head_dim, dtype, seed=0, n_q_tokens=None, q_mult=1.0):
    """Decode queries as uint16 bits, [n_layers][n_agents][n_q_heads][head_dim]
    (or [n_layers][n_agents][n_q_tokens][n_q_heads][head_dim] when n_q_tokens is given)."""
    _, _, _, g_q = _streams(seed, 4)
    shape = (n_layers, n_agents, n_q_heads, head_dim) if n_q_tokens is None else \
        (n_layers, n_agents, n_q_tokens, n_q_heads, head_dim)
    q = g_q.standard_normal(shape, dtype=np.float32) * np.float32(q_mult / 8.0)
    return to_bits(q, dtype)


def gen_suffix(n_layers, n_agents, n_kv_heads, suffix_len, head_dim, dtype, seed=0):
    """Private per-agent uncompressed suffix K/V, [L][A][H][S][d] uint16 bits, same distributions."""
    ss = np.random.SeedSequence(seed).spawn(6)[4:]
    g_k, g_v = [np.random.Generator(np.random.PCG64(s)) for s in ss]
    chan = np.exp(g_k.standard_normal((n_layers, 1, n_kv_heads, 1, head_dim), dtype=np.float32))
    k = g_k.standard_normal((n_layers, n_agents, n_kv_heads, suffix_len, head_dim), dtype=np.float32) * chan
    v = g_v.standard_normal((n_layers, n_agents, n_kv_heads, suffix_len, head_dim), dtype=np.float32)
    return to_bits(k, dtype), to_bits(v, dtype)


def gen_workload(w: Workload, seed=0, n_ctx=None, n_agents=None, q_mult=1.0):
    n_ctx = w.n_ctx if n_ctx is None else n_ctx
    n_agents = w.n_agents if n_agents is None else n_agents
    k, v = gen_kv(w.n_layers, w.n_kv_heads, n_ctx, w.head_dim, w.dtype, seed)
    q = gen_q(w.n_layers, n_agents, w.n_q_heads, w.head_dim, w.dtype, seed, q_mult=q_mult)
    return k, v, q
