"""C-ABI checks that need no GPU: the library loads, exports every symbol
declared in include/*.h, embeds the oracle's codebook bit-for-bit, lays out
the pool as documented and rejects bad arguments before any launch."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import oracle
import serving_q8_encode_gb300 as pk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pk.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return pk.load_library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"POLYKV_API\s+[\w\s\*]+?\b(polykv_\w+)\s*\(", src):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"polykv_pool_create", "polykv_encode", "polykv_attend", "polykv_free"} <= names
    for n in names:
        assert hasattr(lib, n), n


def test_codebook_matches_oracle_bit_for_bit(lib):
    c, b = pk.polykv_codebook()
    c32, b32 = oracle.codebook.codebook_f32()
    assert np.array_equal(np.array(c, np.float32).view(np.uint32), c32.view(np.uint32))
    assert np.array_equal(np.array(b, np.float32).view(np.uint32), b32.view(np.uint32))


def _desc(L=2, H=4, d=128, cap=300, dt=pk.POLYKV_BF16):
    return pk.PoolDesc(L, H, d, cap, dt)


def test_query_mode_and_layout(lib):
    _, req = pk.polykv_pool_create(_desc(), None, 0)
    # fake, never dereferenced 256-aligned address: create only records offsets
    h, _ = pk.polykv_pool_create(_desc(), 1 << 40, req)
    try:
        r = pk.polykv_pool_get_regions(h)
        C = r.capacity_rounded
        assert C == 384 and r.total_bytes == req
        U = 2 * 4
        assert r.k_scales_off - r.k_codes_off >= U * C * 128
        assert r.v_codes_off - r.k_scales_off >= U * C * 4 * 2
        assert r.v_norms_off - r.v_codes_off >= U * C * 48
        assert r.total_bytes - r.v_norms_off >= U * C * 2
        assert r.status_off == 0 and r.v_nmax_off == 256 and r.header_bytes >= 256 + 4 * U
        assert r.k_codes_off >= r.header_bytes
        for off in (r.k_codes_off, r.k_scales_off, r.v_codes_off, r.v_norms_off, r.header_bytes):
            assert off % 256 == 0
    finally:
        pk.polykv_free(h)


@pytest.mark.parametrize("bad", [dict(d=96), dict(d=32), dict(L=0), dict(H=-1), dict(cap=0), dict(dt=7)])
def test_create_rejects_bad_desc(lib, bad):
    kw = dict(L=2, H=4, d=128, cap=300, dt=pk.POLYKV_BF16)
    kw.update(bad)
    with pytest.raises(pk.PolyKVError) as e:
        pk.polykv_pool_create(_desc(**kw), None, 0)
    assert e.value.status in (1, 2)


def test_create_rejects_small_or_misaligned_buffer(lib):
    _, req = pk.polykv_pool_create(_desc(), None, 0)
    with pytest.raises(pk.PolyKVError) as e:
        pk.polykv_pool_create(_desc(), 1 << 40, req - 1)
    assert e.value.status == 3
    with pytest.raises(pk.PolyKVError) as e:
        pk.polykv_pool_create(_desc(), (1 << 40) + 16, req)
    assert e.value.status == 1


def test_call_order_and_argument_errors_before_launch(lib):
    _, req = pk.polykv_pool_create(_desc(), None, 0)
    h, _ = pk.polykv_pool_create(_desc(), 1 << 40, req)
    try:
        # gap after the (empty) encoded prefix
        with pytest.raises(pk.PolyKVError) as e:
            pk.polykv_encode(h, 1 << 20, 1 << 21, 5, 10, None)
        assert e.value.status == 6
        # beyond capacity
        with pytest.raises(pk.PolyKVError) as e:
            pk.polykv_encode(h, 1 << 20, 1 << 21, 0, 301, None)
        assert e.value.status == 1
        # n_tokens == 0 is a no-op
        pk.polykv_encode(h, 0, 0, 0, 0, None)
        # attend before anything is encoded
        with pytest.raises(pk.PolyKVError) as e:
            pk.polykv_attend(h, 1 << 20, 1 << 21, 1, 8, 1, 0.0, None, 0, None)
        assert e.value.status == 6
        with pytest.raises(pk.PolyKVError) as e:
            pk.polykv_attend_workspace_size(h, 1, 6, 1)  # 6 q heads over 4 kv heads
        assert e.value.status == 1
        with pytest.raises(pk.PolyKVError) as e:
            pk.polykv_attend(h, 1 << 20, 1 << 21, 0, 8, 1, 0.0, None, 0, None)
        assert e.value.status == 1
        msg = pk.load_library().polykv_last_error().decode()
        assert "n_agents" in msg
    finally:
        pk.polykv_free(h)


def test_free_null_is_ok(lib):
    pk.polykv_free(None)


def test_attend_ext_struct_matches_header():
    """The binding's polykv_attend_ext mirrors include/polykv.h field by field."""
    import ctypes
    import serving_q8_encode_gb300 as pk
    names = [f[0] for f in pk.AttendExt._fields_]
    hdr = open(os.path.join(ROOT, "include", "polykv.h")).read()
    body = hdr[hdr.index("typedef struct {\n    /* Private per-agent suffix"):hdr.index("} polykv_attend_ext;")]
    import re
    declared = re.findall(r"^\s+(?:const void\*|int64_t)\s+(\w+);", body, re.M)
    assert names == declared
    assert ctypes.sizeof(pk.AttendExt) == 48
