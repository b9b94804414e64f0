"""polykv_attend_static_ws: attention for callers that cannot allocate device memory when they
attend (graph capture elsewhere in the process, allocator-less hosts). It keeps the split
partials in the library's built-in 16 MiB device array instead of a caller workspace; its
output must match polykv_attend's, on consecutive calls that reuse the shared array. This file
is collected last on purpose."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk_torch():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import serving_q8_encode_gb300 as pk
    return pk, torch


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


@pytest.mark.parametrize("L,H,Hq,d,T,A,dtype", [
    (32, 8, 32, 128, 4096, 15, "bf16"),   # Llama-3-8B shape, 15 agents (tensor-core path)
    (2, 32, 32, 64, 1851, 5, "f16"),      # SmolLM2 shape (CUDA-core path)
])
def test_static_workspace_matches_caller_workspace(pk_torch, L, H, Hq, d, T, A, dtype):
    pk, torch = pk_torch
    kb, vb = synth.gen_kv(L, H, T, d, dtype, seed=3)
    pool = pk.Pool(L, H, d, T, dtype)
    pool.encode(_dev(torch, kb), _dev(torch, vb))
    stream = torch.cuda.current_stream().cuda_stream
    ref = None
    for call in range(2):  # two calls in a row: the second reuses the array the first left behind
        qb = synth.gen_q(L, A, Hq, d, dtype, seed=10 + call)
        q = _dev(torch, qb)
        want = pool.attend(q, T)
        got = torch.empty_like(want)
        pk.polykv_attend_static_ws(pool.handle, q.data_ptr(), got.data_ptr(), A, Hq, T, 0.0, stream)
        torch.cuda.synchronize()
        assert pool.status() == 0
        err = (got - want).abs().max().item()
        assert err <= 2e-3, err
        if ref is not None:
            assert not torch.equal(got, ref)  # a fresh result, not the previous call's
        ref = got.clone()


def test_static_workspace_rejects_oversized_arguments(pk_torch):
    pk, torch = pk_torch
    # 512 (layer, kv head) units x 400 query rows each: about 54 MB of partials, above the 16 MiB array
    L, H, d, T, A = 8, 64, 64, 128, 400
    pool = pk.Pool(L, H, d, T, "f16")
    kb = np.zeros((L, H, T, d), np.uint16)
    pool.encode(_dev(torch, kb), _dev(torch, kb))
    q = torch.zeros((L, A, H, d), dtype=torch.int16, device="cuda")
    out = torch.empty((L, A, H, d), dtype=torch.float32, device="cuda")
    with pytest.raises(pk.PolyKVError) as e:
        pk.polykv_attend_static_ws(pool.handle, q.data_ptr(), out.data_ptr(), A, H, T, 0.0,
                                   torch.cuda.current_stream().cuda_stream)
    assert e.value.status == 3 and "16777216" in str(e.value)
