"""Repeated attention calls over one pool must give bit-identical outputs.

The tensor-core path overlaps TMA refills of a shared-memory ring, thread-written
operands and tcgen05 MMAs; an ordering mistake between those shows up first as
rare run-to-run differences (one tile of one unit off), long before it breaks a
tolerance test. Runs at the Llama-3-8B shape (32 layers x 8 kv heads, 4096
tokens, 15 agents x 4 GQA heads), where every CTA crosses a unit boundary."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def test_repeated_calls_are_bit_identical():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import serving_q8_encode_gb300 as pk

    L, H, Hq, d, T, A = 32, 8, 32, 128, 4096, 15
    kb, vb = synth.gen_kv(L, H, T, d, "bf16", seed=3)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    pool = pk.Pool(L, H, d, T, "bf16")
    pool.encode(dev(kb), dev(vb))
    q = dev(synth.gen_q(L, A, Hq, d, "bf16", seed=10))
    ws = torch.empty(pool.workspace_size(A, Hq, T), dtype=torch.uint8, device="cuda")
    ref = pool.attend(q, T, workspace=ws).clone()
    for call in range(24):
        ws.fill_(0xFF)  # NaN patterns: a partial slot read before it is written would show
        got = pool.attend(q, T, workspace=ws)
        torch.cuda.synchronize()
        assert pool.status() == 0
        assert torch.equal(got, ref), f"call {call + 1}: max diff {(got - ref).abs().max().item()}"
