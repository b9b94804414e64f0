"""Bounded device-side waits: a wait that can never complete (the tensor-core
issuer is told to issue nothing) must give up, report through the pool's
status word, free its resources, and leave the context usable. Faults, traps
and hangs are never used."""
import os

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


def test_stalled_wait_times_out_and_context_survives():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import serving_q8_encode_gb300 as pk

    L, H, Hq, d, T, A = 1, 2, 8, 128, 256, 2
    kb, vb = synth.gen_kv(L, H, T, d, "bf16", 5)
    qb = synth.gen_q(L, A, Hq, d, "bf16", 5)
    pool = pk.Pool(L, H, d, T, "bf16")
    pool.encode(torch.from_numpy(kb.view(np.int16)).cuda(), torch.from_numpy(vb.view(np.int16)).cuda())
    q = torch.from_numpy(qb.view(np.int16)).cuda()
    old = os.environ.get("POLYKV_ATTEND_PATH")
    os.environ["POLYKV_ATTEND_PATH"] = "tc"   # the stall hook is the tensor-core kernel's
    os.environ["POLYKV_TEST_STALL"] = "1"
    try:
        pool.attend(q, T)
        torch.cuda.synchronize()
    finally:
        del os.environ["POLYKV_TEST_STALL"]
        if old is None:
            del os.environ["POLYKV_ATTEND_PATH"]
        else:
            os.environ["POLYKV_ATTEND_PATH"] = old
    with pytest.raises(pk.PolyKVError) as e:
        pool.status()
    assert e.value.status == 5  # E_TIMEOUT
    assert pool.status() == 0   # the read cleared it
    # the context is still usable and the next call is correct
    out = pool.attend(q, T)
    torch.cuda.synchronize()
    assert pool.status() == 0
    c32, b32 = oracle.codebook.codebook_f32()
    ref = oracle.attention.attend_pool(qb, "bf16", oracle.attention.encode_pool(kb, vb, "bf16", b32), T, c32)
    assert np.max(np.abs(out.cpu().numpy() - ref)) <= 2e-3
