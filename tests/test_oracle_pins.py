"""Pins for the CPU oracle against facts fixed outside it: a published
quantizer table, the abstract's printed figures, closed forms, invariants,
library routines (scipy) and brute force on tiny inputs. No GPU."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import accounting, attention, codebook, keys, values

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- codebook
def test_lloyd_max_matches_max_1960_table():
    c, b = codebook.lloyd_max_normal()
    rows = _read_golden("max1960_gaussian_8level.txt")
    thr = {int(r[1]): float(r[2]) for r in rows if r[0] == "threshold"}
    out = {int(r[1]): float(r[2]) for r in rows if r[0] == "output"}
    mse = [float(r[2]) for r in rows if r[0] == "mse"][0]
    pos_c = c[4:]
    pos_b = b[3:]
    for i in range(1, 5):
        assert abs(pos_c[i - 1] - out[i]) < 6e-4, (i, pos_c[i - 1], out[i])
        assert abs(pos_b[i - 1] - thr[i]) < 6e-4, (i, pos_b[i - 1], thr[i])
    assert abs(codebook.mse_normal(c, b) - mse) < 2e-5


def test_lloyd_max_centroid_condition_by_quadrature():
    integrate = pytest.importorskip("scipy.integrate")
    c, b = codebook.lloyd_max_normal()
    edges = [-np.inf] + list(b) + [np.inf]
    phi = lambda x: math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)
    for i in range(8):
        num = integrate.quad(lambda x: x * phi(x), edges[i], edges[i + 1], epsabs=1e-13)[0]
        den = integrate.quad(phi, edges[i], edges[i + 1], epsabs=1e-13)[0]
        assert abs(num / den - c[i]) < 1e-8
    # boundaries are midpoints
    assert np.allclose(b, 0.5 * (c[:-1] + c[1:]), atol=0, rtol=0)


def test_lloyd_max_mse_by_quadrature():
    integrate = pytest.importorskip("scipy.integrate")
    c, b = codebook.lloyd_max_normal()
    edges = [-np.inf] + list(b) + [np.inf]
    phi = lambda x: math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)
    tot = sum(integrate.quad(lambda x: (x - c[i]) ** 2 * phi(x), edges[i], edges[i + 1], epsabs=1e-13)[0]
              for i in range(8))
    assert abs(tot - codebook.mse_normal(c, b)) < 1e-9
    assert abs(tot - 0.0345) < 1e-4


def test_lloyd_max_vs_sampled_kmeans():
    rng = np.random.default_rng(123)
    x = np.sort(rng.standard_normal(1_000_000))
    c = np.linspace(-2, 2, 8)
    for _ in range(200):
        bnd = 0.5 * (c[:-1] + c[1:])
        idx = np.searchsorted(bnd, x)
        c = np.array([x[idx == i].mean() for i in range(8)])
    c_lm, _ = codebook.lloyd_max_normal()
    assert np.max(np.abs(c - c_lm)) < 0.01


def test_codebook_f32_symmetric_and_ordered():
    c32, b32 = codebook.codebook_f32()
    assert c32.dtype == np.float32 and b32.dtype == np.float32
    assert np.all(np.diff(c32) > 0) and np.all(np.diff(b32) > 0)
    assert np.array_equal(c32, -c32[::-1])
    assert b32[3] == 0.0
    assert np.all((b32 > c32[:-1]) & (b32 < c32[1:]))


# ---------------------------------------------------------------- q8_0 keys
def test_q8_worked_block():
    rows = _read_golden("q8_0_worked_block.txt")
    x = np.zeros(32, dtype=np.float32)
    want = np.zeros(32, dtype=np.int8)
    for i, r in enumerate(rows):
        x[i] = float(r[0])
        want[i] = int(r[2])
    q, s = keys.quantize_q8_0(x[None, :])
    assert float(s[0, 0]) == 0.0625
    assert np.array_equal(q[0], want)


def _exact_nearest_code(x, s):
    """Exact-rational nearest code with ties away from zero."""
    r = Fraction(float(x)) / Fraction(float(s))
    best = None
    for cand in range(-127, 128):
        err = abs(r - cand)
        key = (err, -abs(cand))
        if best is None or key < best[0]:
            best = (key, cand)
    return best[1], r


def test_q8_bruteforce_exact_rational():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((40, 32)) * np.exp(rng.standard_normal((40, 1)) * 3)).astype(np.float32)
    q, s = keys.quantize_q8_0(x)
    for i in range(x.shape[0]):
        amax = float(np.max(np.abs(x[i])))
        # scale: fp16 of amax/127 via a float64 route (differs only on double-rounding ties)
        s64 = np.float64(amax) / 127.0
        assert abs(float(s[i, 0]) - float(np.float16(s64))) <= 0.0 or \
            abs(float(np.float16(s64)) - float(s[i, 0])) <= np.spacing(np.float16(s64))
        sf = float(s[i, 0])
        for j in range(32):
            code, r = _exact_nearest_code(x[i, j], sf)
            frac = abs(abs(r) - math.floor(abs(r)) - Fraction(1, 2))
            if frac < Fraction(1, 2 ** 20):
                assert abs(int(q[i, j]) - float(r)) <= 0.5 + 1e-6
            else:
                assert int(q[i, j]) == code, (i, j, float(r), q[i, j], code)


def test_q8_roundtrip_bound_and_amax_code():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((2000, 128)) * np.exp(rng.standard_normal((1, 128)))).astype(np.float32)
    q, s = keys.quantize_q8_0(x)
    khat = keys.dequantize_q8_0(q, s)
    sf = np.repeat(s.astype(np.float64), 32, axis=-1)
    err = np.abs(x.astype(np.float64) - khat)
    slack = np.spacing(np.abs(x)).astype(np.float64)
    assert np.all(err <= sf / 2 + slack)
    xb = np.abs(x.reshape(2000, 4, 32))
    qb = np.abs(q.reshape(2000, 4, 32).astype(np.int32))
    arg = np.argmax(xb, axis=-1)
    assert np.all(np.take_along_axis(qb, arg[..., None], -1) == 127)


def test_q8_zero_block():
    q, s = keys.quantize_q8_0(np.zeros((1, 64), np.float32))
    assert np.all(q == 0) and np.all(s == 0)


# ---------------------------------------------------------------- FWHT / values
@pytest.mark.parametrize("d", [8, 64, 128])
def test_fwht_matches_scipy_hadamard(d):
    linalg = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(d)
    v = rng.standard_normal((50, d))
    H = linalg.hadamard(d)
    ref = v @ H.T
    assert np.allclose(values.fwht_f64(v), ref, atol=1e-12)
    got32 = values.fwht_f32_pinned(v.astype(np.float32))
    assert np.allclose(got32, (v.astype(np.float32).astype(np.float64)) @ H.T, atol=1e-4 * math.sqrt(d))


@pytest.mark.parametrize("d", [64, 128])
def test_fwht_self_inverse_and_norm(d):
    rng = np.random.default_rng(1)
    v = rng.standard_normal((100, d))
    y = values.fwht_f64(v) / math.sqrt(d)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(v, axis=1), rtol=1e-12)
    assert np.allclose(values.fwht_f64(y) / math.sqrt(d), v, atol=1e-12)


def test_sumsq_pinned_close_to_float64():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((1000, 128)).astype(np.float32)
    s = values.sumsq_f32_pinned(v).astype(np.float64)
    ref = np.sum(v.astype(np.float64) ** 2, axis=1)
    assert np.all(np.abs(s - ref) <= 1e-5 * ref)


def test_sumsq_pinned_order_by_hand():
    # order matters in fp32: a large group sum absorbs a tiny square only when
    # the tiny one is added after the large one inside the same group.
    v = np.zeros(64, np.float32)
    v[0] = np.float32(2.0 ** 12)          # square 2^24
    v[1] = np.float32(1.0)                # 1 + 2^24 -> rounds back to 2^24 (tie to even)
    v[8] = np.float32(1.0)                # second group: exactly 1
    got = float(values.sumsq_f32_pinned(v[None, :])[0])
    # group0 = 2^24 (the +1 is lost), group1 = 1, tree: 2^24 + 1 -> 2^24
    assert got == 2.0 ** 24


@pytest.mark.parametrize("d", [64, 128])
def test_value_codes_nearest_centroid(d):
    c32, b32 = codebook.codebook_f32()
    rng = np.random.default_rng(5)
    v = rng.standard_normal((3000, d)).astype(np.float32)
    codes, n16, u = values.encode_values(v, b32)
    near = np.argmin(np.abs(u[..., None].astype(np.float64) - c32.astype(np.float64)), axis=-1)
    b = b32.astype(np.float64)
    dist = np.min(np.abs(u[..., None].astype(np.float64) - b), axis=-1)
    ok = (codes == near) | (dist < 1e-6)
    assert np.all(ok)
    # sum of u^2 equals d (norm preservation of H / sqrt(d) after scaling)
    assert np.allclose(np.sum(u.astype(np.float64) ** 2, axis=1), d, rtol=1e-5)
    assert abs(float(np.mean(u))) < 0.01 and abs(float(np.var(u)) - 1.0) < 0.01


def test_value_nmse_gaussian_d128():
    c32, b32 = codebook.codebook_f32()
    rng = np.random.default_rng(6)
    v = rng.standard_normal((4000, 128)).astype(np.float32)
    codes, n16, _ = values.encode_values(v, b32)
    vhat = values.dequantize_values(codes, n16, c32)
    nmse = np.mean(np.sum((vhat - v) ** 2, axis=1) / np.sum(v.astype(np.float64) ** 2, axis=1))
    assert abs(nmse - 0.0345) < 0.003, nmse


def test_value_dequant_norm_identity():
    c32, b32 = codebook.codebook_f32()
    rng = np.random.default_rng(8)
    v = rng.standard_normal((200, 64)).astype(np.float32)
    codes, n16, _ = values.encode_values(v, b32)
    vhat = values.dequantize_values(codes, n16, c32)
    cn = np.linalg.norm(c32.astype(np.float64)[codes], axis=1)
    assert np.allclose(np.linalg.norm(vhat, axis=1), n16.astype(np.float64) / 8.0 * cn, rtol=1e-12)


def test_zero_value_vector():
    c32, b32 = codebook.codebook_f32()
    codes, n16, u = values.encode_values(np.zeros((1, 128), np.float32), b32)
    assert np.all(codes == 4) and float(n16[0]) == 0.0
    assert np.all(values.dequantize_values(codes, n16, c32) == 0)


def _check_pack_worked_group():
    rows = {r[0]: r[1:] for r in _read_golden("pack_worked_group.txt")}
    c0 = np.array([int(x) for x in rows["codes0"]], np.uint8)
    c1 = np.array([int(x) for x in rows["codes1"]], np.uint8)
    want = np.array([int(x, 16) for x in rows["bytes"]], np.uint8).reshape(2, 12)
    got = values.pack_codes(np.stack([c0, c1], axis=-1))      # [32 tokens][2 coordinates]
    assert got.shape == (1, 2, 12)
    assert np.array_equal(got[0], want)


def test_pack_worked_group_and_roundtrip():
    _check_pack_worked_group()
    rng = np.random.default_rng(9)
    c = rng.integers(0, 8, (3, 96, 128)).astype(np.uint8)
    p = values.pack_codes(c)
    assert p.shape == (3, 3, 128, 12)                          # 3 bits per code: 12 bytes per 32 tokens
    assert np.array_equal(values.unpack_codes(p, 128), c)


def test_pack_group_independence():
    """Each 12-byte string depends only on its own coordinate and 32-token group."""
    rng = np.random.default_rng(4)
    c = rng.integers(0, 8, (64, 16)).astype(np.uint8)
    p = values.pack_codes(c)
    c2 = c.copy()
    c2[40, 5] ^= 7                                             # token 40 = group 1, k = 8
    p2 = values.pack_codes(c2)
    diff = np.argwhere(p != p2)
    assert set(map(tuple, diff[:, :2])) == {(1, 5)}
    assert set(diff[:, 2]) == {3}                              # bits 24..26 live in byte 3


# ---------------------------------------------------------------- attention
def _small_pool(T=9, H=2, d=64, seed=0):
    c32, b32 = codebook.codebook_f32()
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((H, T, d)).astype(np.float32)
    v = rng.standard_normal((H, T, d)).astype(np.float32)
    kc, ks = keys.quantize_q8_0(k)
    vc, vn, _ = values.encode_values(v, b32)
    return keys.dequantize_q8_0(kc, ks), values.dequantize_values(vc, vn, c32)


def test_attention_q_zero_is_mean_of_values():
    kh, vh = _small_pool()
    q = np.zeros((3, 4, 64))
    out = attention.attend_layer(q, kh, vh, 0.125)
    for hq in range(4):
        assert np.allclose(out[:, hq], vh[hq // 2].mean(axis=0)[None, :], atol=1e-12)


def test_attention_single_token_returns_its_value():
    kh, vh = _small_pool(T=1)
    rng = np.random.default_rng(1)
    out = attention.attend_layer(rng.standard_normal((2, 2, 64)), kh, vh, 0.125)
    assert np.allclose(out[:, 0], vh[0, 0], atol=1e-12)
    assert np.allclose(out[:, 1], vh[1, 0], atol=1e-12)


def test_attention_dominant_key():
    kh, vh = _small_pool(T=12, H=1)
    q = (kh[0, 5] * 100.0)[None, None, :]
    out = attention.attend_layer(q, kh, vh, 1.0)
    assert np.allclose(out[0, 0], vh[0, 5], atol=1e-9)


def test_attention_constant_values():
    kh, vh = _small_pool(T=7, H=1)
    vconst = np.tile(np.linspace(-1, 1, 64)[None, None, :], (1, 7, 1))
    rng = np.random.default_rng(4)
    out = attention.attend_layer(rng.standard_normal((1, 1, 64)), kh, vconst, 0.3)
    assert np.allclose(out[0, 0], vconst[0, 0], atol=1e-12)


def test_attention_two_token_logistic():
    kh, vh = _small_pool(T=2, H=1)
    rng = np.random.default_rng(5)
    q = rng.standard_normal(64)
    s0, s1 = 0.2 * float(q @ kh[0, 0]), 0.2 * float(q @ kh[0, 1])
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    want = w0 * vh[0, 0] + (1 - w0) * vh[0, 1]
    out = attention.attend_layer(q[None, None, :], kh, vh, 0.2)
    assert np.allclose(out[0, 0], want, atol=1e-12)


def test_attention_gqa_head_mapping():
    # kv head h holds constant value vector h+1; q head hq must read kv head hq // G
    H, G, T, d = 4, 3, 5, 64
    kh = np.random.default_rng(0).standard_normal((H, T, d))
    vh = np.stack([np.full((T, d), h + 1.0) for h in range(H)])
    out = attention.attend_layer(np.random.default_rng(1).standard_normal((2, H * G, d)), kh, vh, 0.1)
    for hq in range(H * G):
        assert np.allclose(out[:, hq], hq // G + 1.0)


def test_attention_permutation_invariance():
    kh, vh = _small_pool(T=10, H=1)
    perm = np.random.default_rng(2).permutation(10)
    q = np.random.default_rng(3).standard_normal((2, 1, 64))
    a = attention.attend_layer(q, kh, vh, 0.125)
    b = attention.attend_layer(q, kh[:, perm], vh[:, perm], 0.125)
    assert np.allclose(a, b, atol=1e-12)


def test_rotated_basis_linearity_identity():
    # sum_t p_t v_hat_t == (1/d) H sum_t p_t n_t C[code_t]
    c32, b32 = codebook.codebook_f32()
    rng = np.random.default_rng(11)
    v = rng.standard_normal((20, 128)).astype(np.float32)
    codes, n16, _ = values.encode_values(v, b32)
    p = rng.random(20)
    vh = values.dequantize_values(codes, n16, c32)
    lhs = p @ vh
    acc = (p * n16.astype(np.float64)) @ c32.astype(np.float64)[codes]
    rhs = values.fwht_f64(acc) / 128.0
    assert np.allclose(lhs, rhs, atol=1e-12)


def test_suffix_equals_concatenated_pool():
    kh, vh = _small_pool(T=6, H=1)
    rng = np.random.default_rng(12)
    sk = rng.standard_normal((2, 1, 3, 64))
    sv = rng.standard_normal((2, 1, 3, 64))
    q = rng.standard_normal((2, 1, 64))
    out = attention.attend_layer(q, kh, vh, 0.125, sk, sv)
    for a in range(2):
        ref = attention.attend_layer(q[a:a + 1], np.concatenate([kh, sk[a]], 1),
                                     np.concatenate([vh, sv[a]], 1), 0.125)
        assert np.allclose(out[a], ref[0], atol=1e-12)


def test_chunk_first_query_sees_pool_plus_itself():
    kh, vh = _small_pool(T=5, H=1)
    rng = np.random.default_rng(13)
    C = 4
    ck = rng.standard_normal((1, C, 1, 64))
    cv = rng.standard_normal((1, C, 1, 64))
    q = rng.standard_normal((1, C, 1, 64))
    out = attention.attend_chunk_layer(q, kh, vh, 0.125, ck, cv)
    for i in range(C):
        ref = attention.attend_layer(q[:, i], np.concatenate([kh, ck[0, :i + 1, :].transpose(1, 0, 2)], 1),
                                     np.concatenate([vh, cv[0, :i + 1, :].transpose(1, 0, 2)], 1), 0.125)
        assert np.allclose(out[0, i], ref[0], atol=1e-12)


# ---------------------------------------------------------------- accounting
def test_abstract_figures():
    g = {r[0]: float(r[1]) for r in _read_golden("polykv_abstract_figures.txt")}
    assert round(accounting.nominal_ratio(), 2) == g["compression_ratio"]
    assert round(100 * accounting.shared_pool_reduction(int(g["agents"]), g["compression_ratio"]), 1) \
        == g["reduction_pct"]
    assert round(g["fp16_cache_gb"] / g["agents"] / g["compression_ratio"], 2) == g["pool_gb"]


def test_exact_ratio_with_overheads():
    assert abs(accounting.exact_ratio(64) - 2.7234) < 1e-4
    assert abs(accounting.exact_ratio(128) - 2.7527) < 1e-4
    # bytes per token-head of the pool format: d + 2*d/32 + 3d/8 + 2
    assert accounting.pool_bytes(1, 1, 1, 128) == 186
    assert accounting.pool_bytes(32, 8, 4096, 128) == 195_035_136


# ---------------------------------------------------------------- planted mistakes
# Each test plants a plausible mistake inside the oracle (monkeypatching one of its steps) and
# checks that a pin above goes red; the pins then pass again with the oracle restored.
def test_planted_fwht_sign_error_is_caught(monkeypatch):
    monkeypatch.setattr(values, "butterfly", lambda a, b: (a + b, b - a))
    with pytest.raises(AssertionError):
        test_fwht_matches_scipy_hadamard(64)
    with pytest.raises(AssertionError):
        test_value_nmse_gaussian_d128()


def test_planted_half_even_rounding_is_caught(monkeypatch):
    monkeypatch.setattr(keys, "round_half_away", np.round)   # numpy rounds ties to even
    with pytest.raises(AssertionError):
        test_q8_worked_block()


def test_planted_pack_bit_order_is_caught(monkeypatch):
    real = np.packbits
    monkeypatch.setattr(values.np, "packbits", lambda a, axis=-1, bitorder="little": real(a, axis=axis, bitorder="big"))
    with pytest.raises(AssertionError):
        _check_pack_worked_group()


def test_planted_gqa_mapping_is_caught(monkeypatch):
    """A query head reading kv head hq % H instead of hq // G fails the GQA pin."""
    monkeypatch.setattr(attention, "kv_head_of", lambda hq, G, H: hq % H)
    with pytest.raises(AssertionError):
        test_attention_gqa_head_mapping()


def test_q8_subnormal_scale_clamp_binds():
    # amax/127 = 1.4 * 2^-24 rounds to the fp16 subnormal 2^-24, so amax / s16 = 177.8 and the
    # definition's clamp to [-127, 127] decides the code of the largest element.
    s_true = np.float32(1.4 * 2.0 ** -24)
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = s_true * np.float32(127.0)
    x[0, 1] = -x[0, 0]
    x[0, 2] = np.float32(2.0 ** -24) * np.float32(50.0)
    q, s = keys.quantize_q8_0(x)
    assert float(s[0, 0]) == 2.0 ** -24
    assert q[0, 0] == 127 and q[0, 1] == -127 and q[0, 2] == 50


def test_attend_pool_chunk_layout_matches_suffix_per_position():
    """attend_pool in chunk mode ([L][A][H][C][d] chunk K/V, q [L][A][C][Hq][d]) equals, for every
    chunk position c, a suffix of the first c+1 chunk tokens (the suffix path is a separate function)."""
    import synth
    c32, b32 = codebook.codebook_f32()
    L, H, Hq, d, T, A, C = 1, 2, 4, 64, 40, 2, 5
    kb, vb = synth.gen_kv(L, H, T, d, "f16", 3)
    pool = attention.encode_pool(kb, vb, "f16", b32)
    qb = synth.gen_q(L, A * C, Hq, d, "f16", 3).reshape(L, A, C, Hq, d)
    ck, cv = synth.gen_suffix(L, A, H, C, d, "f16", 3)
    got = attention.attend_pool(qb, "f16", pool, T, c32, chunk_k_bits=ck, chunk_v_bits=cv)
    for c in range(C):
        ref = attention.attend_pool(np.ascontiguousarray(qb[:, :, c]), "f16", pool, T, c32,
                                    suffix_k_bits=np.ascontiguousarray(ck[:, :, :, :c + 1]),
                                    suffix_v_bits=np.ascontiguousarray(cv[:, :, :, :c + 1]))
        assert np.allclose(got[:, :, c], ref, atol=1e-12, rtol=0)
