"""Multi-agent decode attention over one shared compressed pool, in float64.

PolyKV abstract: one compressed KV pool is written once and N independent
agents read it concurrently ("multi-reader concurrent agent access"). Each
agent's decode query attends over that single pool. Readings taken:
  * standard scaled dot-product attention, default scale 1/sqrt(d);
  * no mask and no positional rotation inside the pool (keys are stored
    after any rotary embedding was applied);
  * query head hq reads kv head hq // (Hq / H) (grouped-query attention);
  * the result is returned in the original (unrotated) basis.
This module is the plain definition: dequantize the pool (keys.py,
values.py), then softmax(q k_hat^T * scale) v_hat by brute force.
"""
from __future__ import annotations

import numpy as np

from . import keys as _keys
from . import values as _values


def attend_rows(qrows: np.ndarray, khat: np.ndarray, vhat: np.ndarray, scale: float,
                causal_limit=None) -> np.ndarray:
    """qrows [R][d], khat/vhat [T][d] (float64) -> [R][d].
    causal_limit[r] (optional) = number of leading keys row r may see."""
    s = (qrows @ khat.T) * scale
    if causal_limit is not None:
        t = np.arange(khat.shape[0])[None, :]
        s = np.where(t < np.asarray(causal_limit)[:, None], s, -np.inf)
    s = s - np.max(s, axis=1, keepdims=True)
    p = np.exp(s)
    p = p / np.sum(p, axis=1, keepdims=True)
    return p @ vhat


def kv_head_of(hq: int, G: int, H: int) -> int:
    """The kv head read by query head hq (grouped-query attention: G query heads per kv head)."""
    return hq // G


def attend_layer(q_l: np.ndarray, khat_l: np.ndarray, vhat_l: np.ndarray, scale: float,
                 suffix_k=None, suffix_v=None) -> np.ndarray:
    """q_l [A][Hq][d]; khat_l, vhat_l [H][T][d]; optional private per-agent
    suffix_k/suffix_v [A][H][S][d] attended together with the pool under one
    softmax. Returns [A][Hq][d] float64."""
    A, Hq, d = q_l.shape
    H = khat_l.shape[0]
    G = Hq // H
    out = np.zeros((A, Hq, d), dtype=np.float64)
    for a in range(A):
        for hq in range(Hq):
            h = kv_head_of(hq, G, H)
            kk, vv = khat_l[h], vhat_l[h]
            if suffix_k is not None:
                kk = np.concatenate([kk, suffix_k[a, h]], axis=0)
                vv = np.concatenate([vv, suffix_v[a, h]], axis=0)
            out[a, hq] = attend_rows(q_l[a, hq][None, :], kk, vv, scale)[0]
    return out


def attend_chunk_layer(q_l: np.ndarray, khat_l: np.ndarray, vhat_l: np.ndarray, scale: float,
                       chunk_k: np.ndarray, chunk_v: np.ndarray) -> np.ndarray:
    """Query-chunk mode: q_l [A][C][Hq][d]; each agent's C query tokens carry
    their own keys/values chunk_k/chunk_v [A][C][H][d], appended after the
    pool; query i sees the whole pool plus chunk positions 0..i.
    Returns [A][C][Hq][d]."""
    A, C, Hq, d = q_l.shape
    H, T = khat_l.shape[0], khat_l.shape[1]
    G = Hq // H
    out = np.zeros((A, C, Hq, d), dtype=np.float64)
    for a in range(A):
        for hq in range(Hq):
            h = kv_head_of(hq, G, H)
            kk = np.concatenate([khat_l[h], chunk_k[a, :, h]], axis=0)
            vv = np.concatenate([vhat_l[h], chunk_v[a, :, h]], axis=0)
            lim = T + 1 + np.arange(C)
            out[a, :, hq] = attend_rows(q_l[a, :, hq], kk, vv, scale, causal_limit=lim)
    return out


def dequantize_pool_layer(k_codes, k_scales, v_codes, v_norms, centroids_f32):
    """Per-layer float64 (k_hat, v_hat) from the unpacked pool fields
    k_codes int8 [H][T][d], k_scales fp16 [H][T][d/32], v_codes uint8 [H][T][d],
    v_norms fp16 [H][T]."""
    return (_keys.dequantize_q8_0(k_codes, k_scales),
            _values.dequantize_values(v_codes, v_norms, centroids_f32))


def attend_pool(q_bits, dtype, pool, n_ctx, centroids_f32, scale=None, layers=None,
                suffix_k_bits=None, suffix_v_bits=None, chunk_k_bits=None, chunk_v_bits=None):
    """Reference output for a whole pool.

    q_bits: uint16 [L][A][Hq][d] (fp16/bf16 bit patterns); pool: dict with
    unpacked fields 'k_codes' [L][H][>=n_ctx][d] int8, 'k_scales' fp16,
    'v_codes' uint8 [L][H][>=n_ctx][d], 'v_norms' fp16 [L][H][>=n_ctx].
    Returns float64 [len(layers)][A][Hq][d].
    Query-chunk mode (chunk_k_bits/chunk_v_bits [L][A][H][C][d]): q_bits is
    [L][A][C][Hq][d] and the result [len(layers)][A][C][Hq][d]."""
    L = q_bits.shape[0]
    d = q_bits.shape[-1]
    scale = (1.0 / np.sqrt(d)) if scale is None else scale
    layers = range(L) if layers is None else layers
    outs = []
    for l in layers:
        kh, vh = dequantize_pool_layer(pool["k_codes"][l, :, :n_ctx], pool["k_scales"][l, :, :n_ctx],
                                       pool["v_codes"][l, :, :n_ctx], pool["v_norms"][l, :, :n_ctx],
                                       centroids_f32)
        q = _keys.bits_to_f32(q_bits[l], dtype).astype(np.float64)
        if chunk_k_bits is not None:
            # [A][H][C][d] -> [A][C][H][d] as attend_chunk_layer takes it
            ck = _keys.bits_to_f32(chunk_k_bits[l], dtype).astype(np.float64).transpose(0, 2, 1, 3)
            cv = _keys.bits_to_f32(chunk_v_bits[l], dtype).astype(np.float64).transpose(0, 2, 1, 3)
            outs.append(attend_chunk_layer(q, kh, vh, scale, ck, cv))
            continue
        sk = sv = None
        if suffix_k_bits is not None:
            sk = _keys.bits_to_f32(suffix_k_bits[l], dtype).astype(np.float64)
            sv = _keys.bits_to_f32(suffix_v_bits[l], dtype).astype(np.float64)
        outs.append(attend_layer(q, kh, vh, scale, sk, sv))
    return np.stack(outs)


def encode_pool(k_bits, v_bits, dtype, boundaries_f32):
    """Oracle encode of K/V bit patterns [L][H][T][d] -> unpacked pool dict
    (plus the packed codes [L][H][ceil(T/32)][d][12] and the pre-quantization u
    for boundary checks)."""
    k = _keys.bits_to_f32(k_bits, dtype)
    kc, ks = _keys.quantize_q8_0(k)
    del k
    v = _keys.bits_to_f32(v_bits, dtype)
    vc, vn, u = _values.encode_values(v, boundaries_f32)
    T = vc.shape[-2]
    pad = (-T) % _values.GROUP   # a partly filled last group: its missing tokens packed as code 0
    vpad = np.concatenate([vc, np.zeros(vc.shape[:-2] + (pad, vc.shape[-1]), np.uint8)], axis=-2) if pad else vc
    return {"k_codes": kc, "k_scales": ks, "v_codes": vc, "v_norms": vn,
            "v_packed": _values.pack_codes(vpad), "u": u}
