"""PolyKV on GB300: a shared, asymmetrically compressed KV pool read by N agents.

Thin Python binding of ``libpolykv.so`` (ctypes). Every step of the hot path
runs in the library's CUDA kernels; this module only marshals arguments
(device pointers from torch tensors, the current torch stream) and raises on
error. PyTorch provides device memory and streams. There is no CPU fallback:
if the library is missing, importing the binding's functions raises.

Low-level functions carry the C ABI's names (``polykv_pool_create``,
``polykv_encode``, ``polykv_attend``, ``polykv_free``, ...). ``Pool`` wraps
them for torch callers.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpolykv.so")

POLYKV_F16 = 0
POLYKV_BF16 = 1
STATUS_NAMES = {0: "OK", 1: "E_INVAL", 2: "E_UNSUPPORTED", 3: "E_BUFFER_TOO_SMALL", 4: "E_CUDA",
                5: "E_TIMEOUT", 6: "E_STATE"}


class PolyKVError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class PoolDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("capacity_tokens", ctypes.c_int64), ("in_dtype", ctypes.c_int)]


class PoolRegions(ctypes.Structure):
    _fields_ = [("capacity_rounded", ctypes.c_int64), ("k_codes_off", ctypes.c_size_t),
                ("k_scales_off", ctypes.c_size_t), ("v_codes_off", ctypes.c_size_t),
                ("v_norms_off", ctypes.c_size_t), ("status_off", ctypes.c_size_t), ("v_nmax_off", ctypes.c_size_t),
                ("header_bytes", ctypes.c_size_t), ("total_bytes", ctypes.c_size_t)]


class AttendExt(ctypes.Structure):
    _fields_ = [("suffix_k", ctypes.c_void_p), ("suffix_v", ctypes.c_void_p), ("suffix_len", ctypes.c_int64),
                ("chunk_k", ctypes.c_void_p), ("chunk_v", ctypes.c_void_p), ("chunk_len", ctypes.c_int64)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libpolykv.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libpolykv.so is not built at {path}; run `python -c \"import __graft_entry__ as g; "
                          f"g.build()\"` (needs nvcc)")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    sigs = {
        "polykv_pool_create": [ctypes.POINTER(PoolDesc), vp, sz, ctypes.POINTER(vp), ctypes.POINTER(sz)],
        "polykv_pool_get_regions": [vp, ctypes.POINTER(PoolRegions)],
        "polykv_encode": [vp, vp, vp, i64, i64, vp],
        "polykv_attend_workspace_size": [vp, i32, i32, i64, ctypes.POINTER(sz)],
        "polykv_attend": [vp, vp, vp, i32, i32, i64, f32, vp, sz, vp],
        "polykv_free": [vp],
        "polykv_codebook": [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)],
        "polykv_pool_status": [vp, vp, ctypes.POINTER(ctypes.c_uint32)],
        "polykv_attend_static_ws": [vp, vp, vp, i32, i32, i64, f32, vp],
        "polykv_attend_ex_workspace_size": [vp, i32, i32, i64, ctypes.POINTER(AttendExt), ctypes.POINTER(sz)],
        "polykv_attend_ex": [vp, vp, vp, i32, i32, i64, f32, ctypes.POINTER(AttendExt), vp, sz, vp],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.polykv_last_error.argtypes = []
    lib.polykv_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        msg = load_library().polykv_last_error().decode(errors="replace")
        raise PolyKVError(status, msg)


# ------------------------------------------------------------------ C ABI, same names
def polykv_pool_create(desc: PoolDesc, dev_buf: int | None, dev_buf_bytes: int):
    """Returns (handle or None in query mode, required_bytes)."""
    lib = load_library()
    out = ctypes.c_void_p()
    req = ctypes.c_size_t()
    _check(lib.polykv_pool_create(ctypes.byref(desc), dev_buf, dev_buf_bytes, ctypes.byref(out), ctypes.byref(req)))
    return (out.value if dev_buf else None), req.value


def polykv_pool_get_regions(handle: int) -> PoolRegions:
    r = PoolRegions()
    _check(load_library().polykv_pool_get_regions(handle, ctypes.byref(r)))
    return r


def polykv_encode(handle: int, k_ptr: int, v_ptr: int, t0: int, n_tokens: int, stream: int | None):
    _check(load_library().polykv_encode(handle, k_ptr, v_ptr, t0, n_tokens, stream))


def polykv_attend_workspace_size(handle: int, n_agents: int, n_q_heads: int, n_ctx: int) -> int:
    b = ctypes.c_size_t()
    _check(load_library().polykv_attend_workspace_size(handle, n_agents, n_q_heads, n_ctx, ctypes.byref(b)))
    return b.value


def polykv_attend(handle: int, q_ptr: int, out_ptr: int, n_agents: int, n_q_heads: int, n_ctx: int,
                  softmax_scale: float, ws_ptr: int | None, ws_bytes: int, stream: int | None):
    _check(load_library().polykv_attend(handle, q_ptr, out_ptr, n_agents, n_q_heads, n_ctx, softmax_scale, ws_ptr,
                                        ws_bytes, stream))


def polykv_attend_static_ws(handle: int, q_ptr: int, out_ptr: int, n_agents: int, n_q_heads: int, n_ctx: int,
                            softmax_scale: float, stream: int | None):
    """polykv_attend with the library's built-in 16 MiB partials array instead of a caller
    workspace (for callers that cannot allocate device memory when they attend)."""
    _check(load_library().polykv_attend_static_ws(handle, q_ptr, out_ptr, n_agents, n_q_heads, n_ctx,
                                                  softmax_scale, stream))


def polykv_pool_status(handle: int, stream: int | None) -> int:
    """Reads and clears the pool's device status word; raises PolyKVError(E_TIMEOUT) if a kernel gave up."""
    f = ctypes.c_uint32()
    _check(load_library().polykv_pool_status(handle, stream, ctypes.byref(f)))
    return f.value


def polykv_attend_ex_workspace_size(handle: int, n_agents: int, n_q_heads: int, n_ctx: int,
                                    ext: AttendExt | None) -> int:
    b = ctypes.c_size_t()
    _check(load_library().polykv_attend_ex_workspace_size(handle, n_agents, n_q_heads, n_ctx,
                                                          ctypes.byref(ext) if ext is not None else None,
                                                          ctypes.byref(b)))
    return b.value


def polykv_attend_ex(handle: int, q_ptr: int, out_ptr: int, n_agents: int, n_q_heads: int, n_ctx: int,
                     softmax_scale: float, ext: AttendExt | None, ws_ptr: int | None, ws_bytes: int,
                     stream: int | None):
    _check(load_library().polykv_attend_ex(handle, q_ptr, out_ptr, n_agents, n_q_heads, n_ctx, softmax_scale,
                                           ctypes.byref(ext) if ext is not None else None, ws_ptr, ws_bytes, stream))


def polykv_free(handle: int | None):
    _check(load_library().polykv_free(handle))


def polykv_codebook():
    c = (ctypes.c_float * 8)()
    b = (ctypes.c_float * 7)()
    _check(load_library().polykv_codebook(c, b))
    return list(c), list(b)


# ------------------------------------------------------------------ torch wrapper
def _require(t, name: str, *, shape=None, elem_bytes=None, dtype=None, device=None):
    """Argument checks before a pointer crosses the C ABI (which sees only addresses and sizes)."""
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if elem_bytes is not None and t.element_size() != elem_bytes:
        raise ValueError(f"{name} must have {elem_bytes}-byte elements (the pool dtype's bits), got {t.dtype}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the pool on {device}")


def _stream_handle(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


class Pool:
    """One shared compressed pool in a torch-allocated device buffer."""

    def __init__(self, n_layers: int, n_kv_heads: int, head_dim: int, capacity_tokens: int, dtype: str = "bf16",
                 device="cuda"):
        import torch
        self.dtype = dtype
        self.desc = PoolDesc(n_layers, n_kv_heads, head_dim, capacity_tokens,
                             POLYKV_BF16 if dtype == "bf16" else POLYKV_F16)
        _, req = polykv_pool_create(self.desc, None, 0)
        self.buf = torch.empty(req, dtype=torch.uint8, device=device)
        self.handle, _ = polykv_pool_create(self.desc, self.buf.data_ptr(), req)
        self.regions = polykv_pool_get_regions(self.handle)
        self._ws = None

    @property
    def torch_dtype(self):
        import torch
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    def close(self):
        if getattr(self, "handle", None):
            polykv_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def encode(self, k, v, t0: int = 0, stream=None):
        """k, v: device tensors [L][H][n][d] (the pool's dtype, or int16/uint16 bits), contiguous."""
        if k.dim() != 4:
            raise ValueError(f"k must be [L][H][n][d], got shape {tuple(k.shape)}")
        L, H, n, d = k.shape
        want = (self.desc.n_layers, self.desc.n_kv_heads, n, self.desc.head_dim)
        _require(k, "k", shape=want, elem_bytes=2, device=self.buf.device)
        _require(v, "v", shape=want, elem_bytes=2, device=self.buf.device)
        polykv_encode(self.handle, k.data_ptr(), v.data_ptr(), t0, n, _stream_handle(stream))

    def status(self, stream=None) -> int:
        return polykv_pool_status(self.handle, _stream_handle(stream))

    def workspace_size(self, n_agents: int, n_q_heads: int, n_ctx: int) -> int:
        return polykv_attend_workspace_size(self.handle, n_agents, n_q_heads, n_ctx)

    def attend(self, q, n_ctx: int, out=None, workspace=None, softmax_scale: float = 0.0, stream=None):
        """q: device [L][A][Hq][d] (pool dtype bits). Returns fp32 out of the same shape."""
        import torch
        if q.dim() != 4:
            raise ValueError(f"q must be [L][A][Hq][d], got shape {tuple(q.shape)}")
        L, A, Hq, d = q.shape
        _require(q, "q", elem_bytes=2, device=self.buf.device)
        if out is None:
            out = torch.empty((L, A, Hq, d), dtype=torch.float32, device=q.device)
        _require(out, "out", shape=(L, A, Hq, d), dtype=torch.float32, device=self.buf.device)
        need = self.workspace_size(A, Hq, n_ctx)
        if workspace is None:
            if self._ws is None or self._ws.numel() < need:
                self._ws = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
            workspace = self._ws
        _require(workspace, "workspace", device=self.buf.device)
        polykv_attend(self.handle, q.data_ptr(), out.data_ptr(), A, Hq, n_ctx, softmax_scale,
                      workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_handle(stream))
        return out

    def attend_with_suffix(self, q, n_ctx: int, suffix_k, suffix_v, out=None, softmax_scale: float = 0.0,
                           stream=None):
        """Pool plus each agent's private uncompressed suffix under one softmax.
        suffix_k/v: device [L][A][H][S][d] (pool dtype bits), contiguous."""
        import torch
        if q.dim() != 4 or suffix_k.dim() != 5:
            raise ValueError("q must be [L][A][Hq][d] and the suffix [L][A][H][S][d]")
        L, A, Hq, d = q.shape
        _require(q, "q", elem_bytes=2, device=self.buf.device)
        sfx_shape = (L, A, self.desc.n_kv_heads, suffix_k.shape[3], d)
        _require(suffix_k, "suffix_k", shape=sfx_shape, elem_bytes=2, device=self.buf.device)
        _require(suffix_v, "suffix_v", shape=sfx_shape, elem_bytes=2, device=self.buf.device)
        ext = AttendExt(suffix_k.data_ptr(), suffix_v.data_ptr(), suffix_k.shape[3])
        if out is None:
            out = torch.empty((L, A, Hq, d), dtype=torch.float32, device=q.device)
        _require(out, "out", shape=(L, A, Hq, d), dtype=torch.float32, device=self.buf.device)
        need = polykv_attend_ex_workspace_size(self.handle, A, Hq, n_ctx, ext)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        polykv_attend_ex(self.handle, q.data_ptr(), out.data_ptr(), A, Hq, n_ctx, softmax_scale, ext, ws.data_ptr(),
                         ws.numel(), _stream_handle(stream))
        return out

    def attend_chunk(self, q, n_ctx: int, chunk_k, chunk_v, out=None, softmax_scale: float = 0.0, stream=None,
                     workspace=None):
        """Query-chunk mode: q device [L][A][C][Hq][d]; chunk_k/v device [L][A][H][C][d] (pool dtype
        bits, contiguous). Query token c of agent a sees the pool plus that agent's chunk tokens 0..c.
        Returns fp32 [L][A][C][Hq][d]."""
        import torch
        if q.dim() != 5:
            raise ValueError(f"q must be [L][A][C][Hq][d], got shape {tuple(q.shape)}")
        L, A, C, Hq, d = q.shape
        _require(q, "q", elem_bytes=2, device=self.buf.device)
        chunk_shape = (L, A, self.desc.n_kv_heads, C, d)
        _require(chunk_k, "chunk_k", shape=chunk_shape, elem_bytes=2, device=self.buf.device)
        _require(chunk_v, "chunk_v", shape=chunk_shape, elem_bytes=2, device=self.buf.device)
        ext = AttendExt(chunk_k=chunk_k.data_ptr(), chunk_v=chunk_v.data_ptr(), chunk_len=C)
        if out is None:
            out = torch.empty((L, A, C, Hq, d), dtype=torch.float32, device=q.device)
        _require(out, "out", shape=(L, A, C, Hq, d), dtype=torch.float32, device=self.buf.device)
        need = polykv_attend_ex_workspace_size(self.handle, A, Hq, n_ctx, ext)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        _require(workspace, "workspace", device=self.buf.device)
        polykv_attend_ex(self.handle, q.data_ptr(), out.data_ptr(), A, Hq, n_ctx, softmax_scale, ext,
                         workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_handle(stream))
        return out

    # -- views of the encoded fields (for inspection and tests)
    def fields(self):
        import torch
        r = self.regions
        L, H, d = self.desc.n_layers, self.desc.n_kv_heads, self.desc.head_dim
        C = r.capacity_rounded
        b = self.buf
        kq = b[r.k_codes_off:r.k_codes_off + L * H * C * d].view(torch.int8).view(L, H, C, d)
        ks = b[r.k_scales_off:r.k_scales_off + L * H * C * (d // 32) * 2].view(torch.float16).view(L, H, C, d // 32)
        # value codes: per 32-token group and coordinate one 12-byte string (token k at bits 3k..3k+2)
        vc = b[r.v_codes_off:r.v_codes_off + L * H * C * (3 * d // 8)].view(L, H, C // 32, d, 12)
        vn = b[r.v_norms_off:r.v_norms_off + L * H * C * 2].view(torch.float16).view(L, H, C)
        return {"k_codes": kq, "k_scales": ks, "v_packed": vc, "v_norms": vn}
