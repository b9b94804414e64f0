"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on
the same seeded inputs. Encode: q8 codes, scales, norms and 3-bit codes
bit-exact (3-bit codes may differ only where the oracle's u lies within
1e-6 * max(|b|, 1) of a boundary b, at most 1e-5 of elements). Attention:
max abs error <= 2e-3 against the float64 oracle over the oracle's pool."""
import os

import numpy as np
import pytest

ERRORS = []   # (case, max abs error, max abs error / max |reference|), printed at the end of the module


def _record(case, err, ref):
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    rel = float(err) / scale if scale > 0 else 0.0
    ERRORS.append((case, float(err), rel))
    print(f"[parity] {case}: max abs err {float(err):.3e}, relative {rel:.3e}")


@pytest.fixture(scope="module", autouse=True)
def _error_table():
    yield
    if ERRORS:
        print("\n[parity] case | max abs err | max abs err / max |ref|")
        for c, e, r in ERRORS:
            print(f"[parity] {c} | {e:.3e} | {r:.3e}")

import oracle
import synth

pytestmark = pytest.mark.gpu

ATOL = 2e-3


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import serving_q8_encode_gb300 as pk
    c32, b32 = oracle.codebook.codebook_f32()
    return pk, torch, c32, b32


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def check_encode(pool, ref, n_tok, t_off=0, b32=None):
    f = {k: v.cpu().numpy() for k, v in pool.fields().items()}
    sl = slice(t_off, t_off + n_tok)
    assert np.array_equal(f["k_codes"][:, :, sl], ref["k_codes"]), "q8 codes differ"
    assert np.array_equal(f["k_scales"][:, :, sl].view(np.uint16), ref["k_scales"].view(np.uint16)), "scales differ"
    assert np.array_equal(f["v_norms"][:, :, sl].view(np.uint16), ref["v_norms"].view(np.uint16)), "norms differ"
    d = ref["v_codes"].shape[-1]
    got = oracle.values.unpack_codes(f["v_packed"], d)[:, :, sl]
    diff = got != ref["v_codes"]
    if diff.any():
        u = ref["u"][diff].astype(np.float64)
        dist = np.min(np.abs(u[:, None] - b32.astype(np.float64)[None, :]) /
                      np.maximum(np.abs(b32.astype(np.float64)), 1.0)[None, :], axis=1)
        assert np.all(dist <= 1e-6), f"{int(diff.sum())} code mismatches away from a boundary"
        assert diff.sum() <= max(1, 1e-5 * diff.size)
    elif t_off % 32 == 0 and n_tok >= 32:
        # whole 32-token groups: the packed bytes themselves
        ng = n_tok // 32
        assert np.array_equal(f["v_packed"][:, :, t_off // 32:t_off // 32 + ng], ref["v_packed"][:, :, :ng])


@pytest.fixture(params=["default", "simt", "tc"])
def path(request):
    """Attention kernel selection: the library's default (the warp-level kernel for few rows per kv
    head, the tensor-core kernel for head_dim 128 and more rows), the CUDA-core path, and the
    tensor-core path where it applies, forced through POLYKV_ATTEND_PATH."""
    old = os.environ.get("POLYKV_ATTEND_PATH")
    if request.param == "default":
        os.environ.pop("POLYKV_ATTEND_PATH", None)
    else:
        os.environ["POLYKV_ATTEND_PATH"] = request.param
    yield request.param
    if old is None:
        os.environ.pop("POLYKV_ATTEND_PATH", None)
    else:
        os.environ["POLYKV_ATTEND_PATH"] = old


def run_case(env, L, H, Hq, d, T, A, dtype, seed=0, q_mult=1.0, n_ctx=None, layers=None, scale=0.0,
             chunks=None):
    pk, torch, c32, b32 = env
    kb, vb = synth.gen_kv(L, H, T, d, dtype, seed)
    qb = synth.gen_q(L, A, Hq, d, dtype, seed, q_mult=q_mult)
    pool = pk.Pool(L, H, d, T, dtype)
    if chunks is None:
        pool.encode(_dev(torch, kb), _dev(torch, vb))
    else:  # append in pieces
        t0 = 0
        for c in chunks:
            pool.encode(_dev(torch, kb[:, :, t0:t0 + c]), _dev(torch, vb[:, :, t0:t0 + c]), t0=t0)
            t0 += c
    n_ctx = T if n_ctx is None else n_ctx
    out = pool.attend(_dev(torch, qb), n_ctx, softmax_scale=scale)
    torch.cuda.synchronize()
    assert pool.status() == 0
    ref_pool = oracle.attention.encode_pool(kb, vb, dtype, b32)
    check_encode(pool, ref_pool, T, 0, b32)
    ref = oracle.attention.attend_pool(qb, dtype, ref_pool, n_ctx, c32,
                                       scale=(scale if scale > 0 else None), layers=layers)
    got = out.cpu().numpy().astype(np.float64)
    if layers is not None:
        got = got[list(layers)]
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    path = os.environ.get("POLYKV_ATTEND_PATH", "default")
    _record(f"L{L} H{H} Hq{Hq} d{d} T{T} A{A} {dtype} q x{q_mult} n_ctx {n_ctx} ({path})", err.max(), ref)
    assert err.max() <= ATOL, f"max abs err {err.max():.3e} (rel {err.max() / np.abs(ref).max():.2e})"
    return err.max()


# ---- the pages' model shapes
def test_smollm2_single_layer_600(env, path):
    run_case(env, 1, 32, 32, 64, 600, 1, "f16")


def test_smollm2_full_stack_1851_5_agents(env, path):
    run_case(env, 24, 32, 32, 64, 1851, 5, "f16", layers=[0, 5, 11, 23])


def test_llama3_8b_4096_15_agents_sampled_layers(env, path):
    run_case(env, 32, 8, 32, 128, 4096, 15, "bf16", layers=[0, 13, 31])


def test_llama3_8b_7194_context(env, path):
    run_case(env, 2, 8, 32, 128, 7194, 15, "bf16")


# ---- ragged and degenerate cases
@pytest.mark.parametrize("T", [1, 31, 33, 64, 65, 129, 257])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_lengths(env, path, T, d):
    run_case(env, 1, 2, 8, d, T, 3, "bf16" if d == 128 else "f16", seed=T)


@pytest.mark.parametrize("A,G", [(1, 1), (2, 4), (15, 4), (20, 4), (33, 2), (7, 1)])
def test_rows_per_kv_head(env, path, A, G):
    run_case(env, 2, 2, 2 * G, 128, 200, A, "bf16", seed=A)


# ---- the warp-level kernel (few rows per kv head): every row count it takes, ragged tails,
# ranges that cross unit boundaries (full layer stacks), peaky queries
@pytest.mark.parametrize("T", [1, 31, 33, 65, 129, 257, 1000])
@pytest.mark.parametrize("d,A,G", [(64, 1, 1), (64, 5, 1), (64, 8, 1), (64, 2, 4), (64, 3, 3), (64, 12, 1),
                                   (64, 16, 1), (128, 1, 1), (128, 1, 4), (128, 2, 2), (128, 5, 1), (128, 3, 2),
                                   (128, 2, 4)])
def test_few_rows_ragged(env, d, A, G, T):
    run_case(env, 2, 3, 3 * G, d, T, A, "f16" if d == 64 else "bf16", seed=T + 7 * A)


@pytest.mark.parametrize("T", [1, 33, 100])
def test_few_rows_many_units_ragged(env, T):
    """A full SmolLM2 layer stack (768 kv-head units) with ragged and tiny contexts: warp ranges that
    cross many unit boundaries."""
    run_case(env, 24, 32, 32, 64, T, 5, "f16", seed=T + 11, layers=[0, 23])


def test_few_rows_many_units_d128(env):
    run_case(env, 80, 8, 32, 128, 65, 1, "bf16", seed=5, layers=[0, 41, 79])


def test_few_rows_llama3_8b_4096_one_agent(env, path):
    run_case(env, 32, 8, 32, 128, 4096, 1, "bf16", layers=[0, 17, 31])


def test_few_rows_llama3_8b_4096_two_agents(env, path):
    """8 query rows per kv head: two score passes over each key group."""
    run_case(env, 32, 8, 32, 128, 4096, 2, "bf16", layers=[0, 17, 31])


def test_few_rows_smollm2_eight_agents_bf16(env):
    run_case(env, 24, 32, 32, 64, 1851, 8, "bf16", layers=[3, 23])


@pytest.mark.parametrize("d,A,G", [(64, 5, 1), (128, 1, 4), (64, 16, 1), (128, 2, 4)])
def test_few_rows_very_peaky(env, path, d, A, G):
    run_case(env, 4, 8, 8 * G, d, 1500, A, "f16" if d == 64 else "bf16", q_mult=40.0)


def test_peaky_queries_online_rescale(env, path):
    run_case(env, 2, 4, 16, 128, 1000, 4, "bf16", q_mult=8.0)


def test_very_peaky_queries(env):
    run_case(env, 1, 2, 8, 64, 700, 3, "f16", q_mult=40.0)


def test_very_peaky_queries_d128(env, path):
    """q x 40 at head_dim 128: one key dominates each softmax, so the fp16 rounding of the
    probabilities and of the value centroids decides the error (tensor-core path by default)."""
    run_case(env, 1, 4, 16, 128, 1500, 4, "bf16", q_mult=40.0)


def test_very_peaky_queries_llama_shape(env):
    """q x 40 on the full 15-agent Llama-3-8B row count (60 rows per kv head), two layers."""
    run_case(env, 2, 8, 32, 128, 4096, 15, "bf16", q_mult=40.0)


def test_zero_queries_give_mean(env, path):
    run_case(env, 1, 2, 8, 128, 300, 2, "bf16", q_mult=0.0)


def test_custom_softmax_scale(env):
    run_case(env, 1, 4, 4, 64, 150, 2, "f16", scale=0.37)


def test_partial_context_and_append(env, path):
    run_case(env, 2, 2, 8, 128, 500, 3, "bf16", n_ctx=333, chunks=[100, 1, 199, 200])


def test_encode_overwrite_in_place(env):
    pk, torch, c32, b32 = env
    L, H, d, T = 1, 2, 128, 64
    k1, v1 = synth.gen_kv(L, H, T, d, "bf16", 1)
    k2, v2 = synth.gen_kv(L, H, 16, d, "bf16", 2)
    pool = pk.Pool(L, H, d, T, "bf16")
    pool.encode(_dev(torch, k1), _dev(torch, v1))
    pool.encode(_dev(torch, k2), _dev(torch, v2), t0=10)
    torch.cuda.synchronize()
    k = k1.copy()
    v = v1.copy()
    k[:, :, 10:26] = k2
    v[:, :, 10:26] = v2
    check_encode(pool, oracle.attention.encode_pool(k, v, "bf16", b32), T, 0, b32)


def test_zero_value_vectors_and_constant_keys(env):
    pk, torch, c32, b32 = env
    L, H, d, T = 1, 1, 64, 40
    kb = np.zeros((L, H, T, d), np.uint16)
    vb = np.zeros((L, H, T, d), np.uint16)
    kb[..., 5:9, :] = synth.f32_to_f16_bits(np.full((1, 1, 4, d), 0.5, np.float32))
    pool = pk.Pool(L, H, d, T, "f16")
    pool.encode(_dev(torch, kb), _dev(torch, vb))
    qb = synth.gen_q(L, 2, 2, d, "f16", 3)
    out = pool.attend(_dev(torch, qb), T)
    torch.cuda.synchronize()
    check_encode(pool, oracle.attention.encode_pool(kb, vb, "f16", b32), T, 0, b32)
    assert np.all(out.cpu().numpy() == 0.0)


def test_two_pools_interleaved_streams(env):
    pk, torch, c32, b32 = env
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    L, H, Hq, d, T, A = 1, 4, 16, 128, 300, 2
    kb, vb = synth.gen_kv(L, H, T, d, "bf16", 9)
    qb = synth.gen_q(L, A, Hq, d, "bf16", 9)
    pool = pk.Pool(L, H, d, T, "bf16")
    pool.encode(_dev(torch, kb), _dev(torch, vb))
    torch.cuda.synchronize()
    q = _dev(torch, qb)
    ws1 = torch.empty(pool.workspace_size(A, Hq, T), dtype=torch.uint8, device="cuda")
    ws2 = torch.empty_like(ws1)
    with torch.cuda.stream(s1):
        o1 = pool.attend(q, T, workspace=ws1, stream=s1)
    with torch.cuda.stream(s2):
        o2 = pool.attend(q, T, workspace=ws2, stream=s2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_tiny_key_blocks_subnormal_scales(env):
    """Blocks whose scale amax/127 falls into (or below) the fp16 subnormal range:
    zero scales, and scales rounded far below amax/127 where the [-127, 127] clamp binds."""
    pk, torch, c32, b32 = env
    L, H, d, T = 1, 2, 128, 96
    rng = np.random.default_rng(21)
    k = rng.standard_normal((L, H, T, d)).astype(np.float32)
    mags = np.array([1e-9, 3e-8, 2e-7, 1e-6, 1e-5, 1.0], np.float32)
    k *= mags[rng.integers(0, len(mags), (L, H, T, d // 32))].repeat(32, axis=-1)
    kb = synth.f32_to_bf16_bits(k)
    vb = synth.f32_to_bf16_bits(rng.standard_normal((L, H, T, d)).astype(np.float32))
    pool = pk.Pool(L, H, d, T, "bf16")
    pool.encode(_dev(torch, kb), _dev(torch, vb))
    torch.cuda.synchronize()
    ref = oracle.attention.encode_pool(kb, vb, "bf16", b32)
    assert np.any(np.abs(ref["k_codes"].astype(int)) == 127)
    check_encode(pool, ref, T, 0, b32)


def test_non_finite_key_blocks(env):
    """A key block holding an inf or a NaN gets a non-finite scale and all-zero codes (the
    oracle's reading); every other block and all values stay bit-exact."""
    pk, torch, c32, b32 = env
    L, H, d, T = 1, 1, 128, 8
    rng = np.random.default_rng(5)
    k = rng.standard_normal((L, H, T, d)).astype(np.float32)
    k[0, 0, 2, 32 + 7] = np.inf
    k[0, 0, 5, 96 + 30] = np.nan
    k[0, 0, 6, 3] = -np.inf
    kb = synth.f32_to_bf16_bits(k)
    vb = synth.f32_to_bf16_bits(rng.standard_normal((L, H, T, d)).astype(np.float32))
    pool = pk.Pool(L, H, d, T, "bf16")
    pool.encode(_dev(torch, kb), _dev(torch, vb))
    torch.cuda.synchronize()
    ref = oracle.attention.encode_pool(kb, vb, "bf16", b32)
    f = {n: x.cpu().numpy()[:, :, :T] for n, x in pool.fields().items() if n != "v_packed"}
    for (t, blk) in ((2, 1), (5, 3), (6, 0)):
        assert not np.isfinite(ref["k_scales"][0, 0, t, blk]) and not np.isfinite(f["k_scales"][0, 0, t, blk])
        assert np.isnan(ref["k_scales"][0, 0, t, blk]) == np.isnan(f["k_scales"][0, 0, t, blk])
        assert np.all(f["k_codes"][0, 0, t, 32 * blk:32 * blk + 32] == 0)
    fin = np.isfinite(ref["k_scales"])
    assert np.array_equal(f["k_scales"][fin].view(np.uint16), ref["k_scales"][fin].view(np.uint16))
    assert np.array_equal(f["k_codes"], ref["k_codes"])
    got_codes = oracle.values.unpack_codes(pool.fields()["v_packed"].cpu().numpy(), d)[:, :, :T]
    assert np.array_equal(got_codes, ref["v_codes"])
    assert np.array_equal(f["v_norms"].view(np.uint16), ref["v_norms"].view(np.uint16))


# ---- pool + private per-agent suffix under one softmax
def run_suffix_case(env, L, H, Hq, d, T, A, S, dtype, seed=0, q_mult=1.0):
    pk, torch, c32, b32 = env
    kb, vb = synth.gen_kv(L, H, T, d, dtype, seed)
    qb = synth.gen_q(L, A, Hq, d, dtype, seed, q_mult=q_mult)
    sk, sv = synth.gen_suffix(L, A, H, S, d, dtype, seed)
    pool = pk.Pool(L, H, d, T, dtype)
    pool.encode(_dev(torch, kb), _dev(torch, vb))
    out = pool.attend_with_suffix(_dev(torch, qb), T, _dev(torch, sk), _dev(torch, sv))
    torch.cuda.synchronize()
    assert pool.status() == 0
    ref_pool = oracle.attention.encode_pool(kb, vb, dtype, b32)
    ref = oracle.attention.attend_pool(qb, dtype, ref_pool, T, c32, suffix_k_bits=sk, suffix_v_bits=sv)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
    path = os.environ.get("POLYKV_ATTEND_PATH", "default")
    _record(f"suffix L{L} H{H} Hq{Hq} d{d} T{T} A{A} S{S} {dtype} q x{q_mult} ({path})", err.max(), ref)
    assert err.max() <= ATOL, f"max abs err {err.max():.3e}"


def test_suffix_llama3_8b_7194_pool_256_private(env, path):
    run_suffix_case(env, 2, 8, 32, 128, 7194, 15, 256, "bf16")


@pytest.mark.parametrize("S", [1, 33, 300])
def test_suffix_ragged_lengths(env, path, S):
    run_suffix_case(env, 1, 4, 16, 128, 200, 3, S, "bf16", seed=S)


def test_suffix_smollm2_mha_fp16(env, path):
    run_suffix_case(env, 2, 32, 32, 64, 600, 2, 64, "f16")


def test_suffix_peaky(env, path):
    run_suffix_case(env, 1, 2, 8, 128, 500, 2, 128, "bf16", q_mult=8.0)


def test_suffix_very_peaky(env):
    """q x 40: one suffix or pool key takes almost all the weight (the suffix's probabilities go into the
    value MMA as a high and a low part; this is where their rounding would show)."""
    run_suffix_case(env, 1, 2, 8, 128, 500, 2, 128, "bf16", q_mult=40.0)


def test_suffix_long_fp16_d64(env):
    """A 1,000-token suffix: each of the four warps of a unit runs many 16-token steps (d = 64, f16)."""
    run_suffix_case(env, 1, 8, 32, 64, 300, 3, 1000, "f16", seed=4)


def test_suffix_sixteen_rows_per_kv_head(env):
    """16 query heads per kv head: more rows than the warp-level suffix kernel takes (CUDA-core kernel)."""
    run_suffix_case(env, 1, 1, 16, 128, 300, 2, 40, "bf16", seed=6)


# ---- query-chunk mode: C query tokens per agent, each with its own key/value, causal inside the chunk
def run_chunk_case(env, L, H, Hq, d, T, A, C, dtype, seed=0, q_mult=1.0):
    pk, torch, c32, b32 = env
    kb, vb = synth.gen_kv(L, H, T, d, dtype, seed)
    qb = synth.gen_q(L, A * C, Hq, d, dtype, seed, q_mult=q_mult).reshape(L, A, C, Hq, d)
    ck, cv = synth.gen_suffix(L, A, H, C, d, dtype, seed)   # [L][A][H][C][d]
    pool = pk.Pool(L, H, d, T, dtype)
    pool.encode(_dev(torch, kb), _dev(torch, vb))
    out = pool.attend_chunk(_dev(torch, qb), T, _dev(torch, ck), _dev(torch, cv))
    torch.cuda.synchronize()
    assert pool.status() == 0
    ref_pool = oracle.attention.encode_pool(kb, vb, dtype, b32)
    ref = oracle.attention.attend_pool(qb, dtype, ref_pool, T, c32, chunk_k_bits=ck, chunk_v_bits=cv)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
    path = os.environ.get("POLYKV_ATTEND_PATH", "default")
    _record(f"chunk L{L} H{H} Hq{Hq} d{d} T{T} A{A} C{C} {dtype} q x{q_mult} ({path})", err.max(), ref)
    assert err.max() <= ATOL, f"max abs err {err.max():.3e}"


def test_chunk_64_tokens_llama3_8b_shape(env, path):
    run_chunk_case(env, 1, 8, 32, 128, 1024, 2, 64, "bf16")


def test_chunk_llama3_8b_4096_15_agents_64_tokens(env):
    """The query-chunk sweep shape: 4,096-token pool, 15 agents x 64 causal query tokens x 4 GQA
    heads = 3,840 rows per kv head (60 row groups), one layer."""
    run_chunk_case(env, 1, 8, 32, 128, 4096, 15, 64, "bf16")


@pytest.mark.parametrize("C", [1, 2, 33, 65, 130])
def test_chunk_ragged_lengths(env, path, C):
    run_chunk_case(env, 1, 2, 8, 128, 300, 2, C, "bf16", seed=C)


def test_chunk_smollm2_mha_fp16(env, path):
    run_chunk_case(env, 1, 32, 32, 64, 600, 1, 16, "f16")


def test_chunk_peaky(env, path):
    run_chunk_case(env, 1, 2, 8, 128, 500, 2, 32, "bf16", q_mult=8.0)


def test_chunk_very_peaky(env):
    """q x 40 in chunk mode: the causal part's probabilities go into the value MMA as high and low parts."""
    run_chunk_case(env, 1, 2, 8, 128, 500, 2, 48, "bf16", q_mult=40.0)


def test_chunk_sixteen_rows_per_kv_head(env):
    """16 query heads per kv head: more rows per chunk position than the warp-level kernel takes."""
    run_chunk_case(env, 1, 1, 16, 128, 300, 2, 20, "bf16", seed=8)


def test_chunk_of_one_equals_one_token_suffix(env):
    """A chunk of length 1 is a one-token private suffix (same keys/values, same softmax)."""
    pk, torch, c32, b32 = env
    L, H, Hq, d, T, A = 1, 2, 8, 128, 200, 3
    kb, vb = synth.gen_kv(L, H, T, d, "bf16", 5)
    qb = synth.gen_q(L, A, Hq, d, "bf16", 5)
    sk, sv = synth.gen_suffix(L, A, H, 1, d, "bf16", 5)
    pool = pk.Pool(L, H, d, T, "bf16")
    pool.encode(_dev(torch, kb), _dev(torch, vb))
    a = pool.attend_with_suffix(_dev(torch, qb), T, _dev(torch, sk), _dev(torch, sv))
    b = pool.attend_chunk(_dev(torch, qb).view(L, A, 1, Hq, d), T, _dev(torch, sk), _dev(torch, sv))
    torch.cuda.synchronize()
    assert (a - b.view(L, A, Hq, d)).abs().max().item() <= 1e-5
