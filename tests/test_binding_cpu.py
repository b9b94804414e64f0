"""The torch-facing binding's argument checks (no GPU): valid calls in the shapes the GPU tests and
the benchmark use reach the C ABI wrappers unchanged; malformed tensors are rejected with
ValueError before any pointer crosses the ABI. The ABI wrappers are replaced by recorders."""
import pytest

torch = pytest.importorskip("torch")
import serving_q8_encode_gb300 as pk  # noqa: E402

L, H, Hq, d, T, A = 2, 4, 8, 128, 300, 3


@pytest.fixture()
def pool(monkeypatch):
    calls = []
    monkeypatch.setattr(pk, "_stream_handle", lambda stream: 0)
    monkeypatch.setattr(pk, "polykv_encode", lambda *a: calls.append(("encode", a)))
    monkeypatch.setattr(pk, "polykv_attend", lambda *a: calls.append(("attend", a)))
    monkeypatch.setattr(pk, "polykv_attend_ex", lambda *a: calls.append(("attend_ex", a)))
    monkeypatch.setattr(pk, "polykv_attend_workspace_size", lambda *a: 1024)
    monkeypatch.setattr(pk, "polykv_attend_ex_workspace_size", lambda *a: 2048)
    p = pk.Pool.__new__(pk.Pool)
    p.dtype = "bf16"
    p.desc = pk.PoolDesc(L, H, d, T, pk.POLYKV_BF16)
    p.buf = torch.empty(16, dtype=torch.uint8)
    p.handle = None
    p._ws = None
    p.calls = calls
    return p


def _bits(*shape):
    return torch.zeros(shape, dtype=torch.int16)


def test_valid_calls_reach_the_abi(pool):
    pool.encode(_bits(L, H, T, d), _bits(L, H, T, d))
    out = pool.attend(_bits(L, A, Hq, d), T)
    assert out.shape == (L, A, Hq, d) and out.dtype == torch.float32
    pool.attend(_bits(L, A, Hq, d), T, out=torch.empty(L, A, Hq, d), workspace=torch.empty(1024, dtype=torch.uint8))
    pool.attend_with_suffix(_bits(L, A, Hq, d), T, _bits(L, A, H, 16, d), _bits(L, A, H, 16, d))
    C = 5
    pool.attend_chunk(_bits(L, A, C, Hq, d), T, _bits(L, A, H, C, d), _bits(L, A, H, C, d))
    pool.attend_chunk(_bits(L, A * 1, Hq, d).view(L, A, 1, Hq, d), T, _bits(L, A, H, 1, d), _bits(L, A, H, 1, d))
    kinds = [c[0] for c in pool.calls]
    assert kinds == ["encode", "attend", "attend", "attend_ex", "attend_ex", "attend_ex"]
    # the encode is passed (t0, n_tokens) = (0, T)
    assert pool.calls[0][1][3:5] == (0, T)


@pytest.mark.parametrize("case", ["k_noncontig", "k_4byte", "k_wrong_heads", "v_shape"])
def test_encode_rejects_malformed(pool, case):
    k, v = _bits(L, H, T, d), _bits(L, H, T, d)
    if case == "k_noncontig":
        k = _bits(L, H, d, T).transpose(2, 3)
    elif case == "k_4byte":
        k = torch.zeros(L, H, T, d, dtype=torch.float32)
    elif case == "k_wrong_heads":
        k, v = _bits(L, H + 1, T, d), _bits(L, H + 1, T, d)
    elif case == "v_shape":
        v = _bits(L, H, T - 1, d)
    with pytest.raises(ValueError):
        pool.encode(k, v)
    assert pool.calls == []


@pytest.mark.parametrize("case", ["q_noncontig", "q_rank", "out_dtype", "out_shape"])
def test_attend_rejects_malformed(pool, case):
    q, out = _bits(L, A, Hq, d), torch.empty(L, A, Hq, d)
    if case == "q_noncontig":
        q = _bits(L, A, d, Hq).transpose(2, 3)
    elif case == "q_rank":
        q = _bits(L, A, Hq * d)
    elif case == "out_dtype":
        out = torch.empty(L, A, Hq, d, dtype=torch.float16)
    elif case == "out_shape":
        out = torch.empty(L, A, Hq, d + 1)
    with pytest.raises(ValueError):
        pool.attend(q, T, out=out)
    assert pool.calls == []


def test_suffix_and_chunk_shapes_checked(pool):
    with pytest.raises(ValueError):   # suffix kv-head count must be the pool's
        pool.attend_with_suffix(_bits(L, A, Hq, d), T, _bits(L, A, H + 1, 16, d), _bits(L, A, H + 1, 16, d))
    with pytest.raises(ValueError):   # chunk length must match the query chunk
        pool.attend_chunk(_bits(L, A, 4, Hq, d), T, _bits(L, A, H, 5, d), _bits(L, A, H, 5, d))
    assert pool.calls == []
