"""Python binding of the R-SWA C ABI (librswa.so).

Argument marshalling only: every entry point converts torch tensors to device
pointers and calls the function of the same name in the shared library, which
does all of the work in CUDA kernels.  There is no Python or CPU fallback: if
the library is missing, ``load()`` raises.

Layouts (see include/rswa.h): prefill tensors are token-major packed rows
``[sum_b (m_b + T)][H][d]``; per-step tensors are ``[B][H][d]``; ``lse`` is
``[B][H]`` float32.
"""

from __future__ import annotations

import ctypes
import os

__all__ = [
    "RswaError", "load", "library_path", "declared_symbols",
    "RSWA_F32", "RSWA_BF16",
    "rswa_strerror", "rswa_cache_footprint", "rswa_cache_create",
    "rswa_cache_footprint_gqa", "rswa_cache_create_gqa", "rswa_prefill_varlen",
    "rswa_cache_destroy", "rswa_prefill", "rswa_append_kv",
    "rswa_decode_step", "rswa_decode_step_fused",
    "rswa_decode_step_fused_static", "rswa_decode_block", "rswa_cache_bytes",
    "rswa_cache_len", "rswa_cache_get_t", "rswa_cache_set_t",
    "rswa_sync_status", "rswa_debug_fail_next_cuda",
    "rswa_debug_set_wait_limit_ns", "rswa_cache_kv_offsets",
    "RswaCache",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
RSWA_F32, RSWA_BF16 = 0, 1
_LIB = None

_c_i64 = ctypes.c_int64
_c_int = ctypes.c_int
_c_vp = ctypes.c_void_p
_c_size = ctypes.c_size_t

_SIGNATURES = {
    "rswa_strerror": (ctypes.c_char_p, [_c_int]),
    "rswa_cache_footprint": (_c_int, [_c_i64, _c_i64, _c_int, _c_int, _c_int,
                                      _c_int, ctypes.POINTER(_c_size)]),
    "rswa_cache_create": (_c_int, [_c_i64, _c_i64, _c_int, _c_int, _c_int,
                                   _c_int, _c_vp, _c_size,
                                   ctypes.POINTER(_c_vp)]),
    "rswa_cache_footprint_gqa": (_c_int, [_c_i64, _c_i64, _c_int, _c_int, _c_int,
                                          _c_int, _c_int, ctypes.POINTER(_c_size)]),
    "rswa_cache_create_gqa": (_c_int, [_c_i64, _c_i64, _c_int, _c_int, _c_int,
                                       _c_int, _c_int, _c_vp, _c_size,
                                       ctypes.POINTER(_c_vp)]),
    "rswa_prefill_varlen": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                     ctypes.POINTER(_c_i64), ctypes.POINTER(_c_i64),
                                     _c_vp]),
    "rswa_cache_destroy": (_c_int, [_c_vp]),
    "rswa_prefill": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                              ctypes.POINTER(_c_i64), _c_i64, _c_vp]),
    "rswa_append_kv": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp]),
    "rswa_decode_step": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp]),
    "rswa_decode_step_fused": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                        _c_vp, _c_vp]),
    "rswa_decode_step_fused_static": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp,
                                               _c_vp, _c_vp, _c_vp]),
    "rswa_decode_block": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_vp,
                                   _c_vp, _c_vp]),
    "rswa_cache_bytes": (_c_int, [_c_vp, _c_int, ctypes.POINTER(_c_size)]),
    "rswa_cache_len": (_c_int, [_c_vp, _c_int, ctypes.POINTER(_c_i64)]),
    "rswa_cache_get_t": (_c_int, [_c_vp, _c_int, ctypes.POINTER(_c_i64)]),
    "rswa_cache_set_t": (_c_int, [_c_vp, ctypes.POINTER(_c_i64), _c_vp]),
    "rswa_sync_status": (_c_int, [_c_vp]),
    "rswa_cache_kv_offsets": (_c_int, [_c_vp, ctypes.POINTER(_c_size),
                                       ctypes.POINTER(_c_size)]),
    "rswa_debug_fail_next_cuda": (None, [_c_int]),
    "rswa_debug_set_wait_limit_ns": (None, [ctypes.c_uint64]),
}


class RswaError(RuntimeError):
    """A non-zero rswa_status returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        msg = load().rswa_strerror(status).decode()
        super().__init__(f"{where}: status {status} ({msg})")


def library_path() -> str:
    return os.path.join(_HERE, "librswa.so")


def declared_symbols() -> list:
    """Names declared RSWA_API in include/rswa.h."""
    import re
    with open(os.path.join(_ROOT, "include", "rswa.h")) as f:
        text = f.read()
    return re.findall(r"RSWA_API\s+[\w\s\*]+?\b(rswa_\w+)\s*\(", text)


def load():
    """Load librswa.so (built by ``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _check(status: int, where: str) -> None:
    if status != 0:
        raise RswaError(status, where)


def _ptr(t):
    """Device pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def rswa_strerror(status: int) -> str:
    return load().rswa_strerror(status).decode()


def rswa_debug_fail_next_cuda(count: int) -> None:
    load().rswa_debug_fail_next_cuda(count)


def rswa_debug_set_wait_limit_ns(ns: int) -> None:
    load().rswa_debug_set_wait_limit_ns(int(ns))


def rswa_cache_footprint(m, n, heads, head_dim, batch, dtype) -> int:
    out = _c_size(0)
    _check(load().rswa_cache_footprint(m, n, heads, head_dim, batch, dtype,
                                       ctypes.byref(out)),
           "rswa_cache_footprint")
    return out.value


def rswa_cache_create(m, n, heads, head_dim, batch, dtype, buf):
    """Create a cache over the uint8 CUDA tensor ``buf``; returns the handle."""
    h = _c_vp()
    _check(load().rswa_cache_create(m, n, heads, head_dim, batch, dtype,
                                    _ptr(buf), buf.numel() * buf.element_size(),
                                    ctypes.byref(h)),
           "rswa_cache_create")
    return h.value


def rswa_cache_footprint_gqa(m, n, heads, kv_heads, head_dim, batch,
                             dtype) -> int:
    out = _c_size(0)
    _check(load().rswa_cache_footprint_gqa(m, n, heads, kv_heads, head_dim,
                                           batch, dtype, ctypes.byref(out)),
           "rswa_cache_footprint_gqa")
    return out.value


def rswa_cache_create_gqa(m, n, heads, kv_heads, head_dim, batch, dtype, buf):
    h = _c_vp()
    _check(load().rswa_cache_create_gqa(m, n, heads, kv_heads, head_dim, batch,
                                        dtype, _ptr(buf),
                                        buf.numel() * buf.element_size(),
                                        ctypes.byref(h)),
           "rswa_cache_create_gqa")
    return h.value


def rswa_cache_destroy(handle) -> None:
    _check(load().rswa_cache_destroy(handle), "rswa_cache_destroy")


def rswa_prefill(handle, Q, K, V, O, m_per_seq, T, stream=None) -> None:
    arr = (_c_i64 * len(m_per_seq))(*[int(x) for x in m_per_seq])
    _check(load().rswa_prefill(handle, _ptr(Q), _ptr(K), _ptr(V), _ptr(O), arr,
                               int(T), _stream(stream)),
           "rswa_prefill")


def rswa_prefill_varlen(handle, Q, K, V, O, m_per_seq, t_per_seq,
                        stream=None) -> None:
    marr = (_c_i64 * len(m_per_seq))(*[int(x) for x in m_per_seq])
    tarr = (_c_i64 * len(t_per_seq))(*[int(x) for x in t_per_seq])
    _check(load().rswa_prefill_varlen(handle, _ptr(Q), _ptr(K), _ptr(V),
                                      _ptr(O), marr, tarr, _stream(stream)),
           "rswa_prefill_varlen")


def rswa_append_kv(handle, k, v, stream=None) -> None:
    _check(load().rswa_append_kv(handle, _ptr(k), _ptr(v), _stream(stream)),
           "rswa_append_kv")


def rswa_decode_step(handle, q, o, lse=None, stream=None) -> None:
    _check(load().rswa_decode_step(handle, _ptr(q), _ptr(o), _ptr(lse),
                                   _stream(stream)),
           "rswa_decode_step")


def rswa_decode_step_fused(handle, q, k, v, o, lse=None, stream=None) -> None:
    _check(load().rswa_decode_step_fused(handle, _ptr(q), _ptr(k), _ptr(v),
                                         _ptr(o), _ptr(lse), _stream(stream)),
           "rswa_decode_step_fused")


def rswa_decode_step_fused_static(handle, q, k, v, o, lse=None,
                                  stream=None) -> None:
    """rswa_decode_step_fused with its split-K scratch in the library's fixed
    4 MiB device array instead of the cache buffer: the call allocates
    nothing (for callers that must not allocate device memory once decoding
    runs).  Overlapping calls race on that array."""
    _check(load().rswa_decode_step_fused_static(handle, _ptr(q), _ptr(k),
                                                _ptr(v), _ptr(o), _ptr(lse),
                                                _stream(stream)),
           "rswa_decode_step_fused_static")


def rswa_decode_block(handle, q, k, v, o, lse=None, stream=None) -> None:
    """q, k, v, o: [B][block][H][d]; lse: [B][block][H] or None."""
    _check(load().rswa_decode_block(handle, _ptr(q), _ptr(k), _ptr(v),
                                    int(q.shape[1]), _ptr(o), _ptr(lse),
                                    _stream(stream)),
           "rswa_decode_block")


def rswa_cache_bytes(handle, b: int) -> int:
    out = _c_size(0)
    _check(load().rswa_cache_bytes(handle, b, ctypes.byref(out)),
           "rswa_cache_bytes")
    return out.value


def rswa_cache_len(handle, b: int) -> int:
    out = _c_i64(0)
    _check(load().rswa_cache_len(handle, b, ctypes.byref(out)), "rswa_cache_len")
    return out.value


def rswa_cache_get_t(handle, b: int) -> int:
    out = _c_i64(0)
    _check(load().rswa_cache_get_t(handle, b, ctypes.byref(out)),
           "rswa_cache_get_t")
    return out.value


def rswa_cache_set_t(handle, t_per_seq, stream=None) -> None:
    arr = (_c_i64 * len(t_per_seq))(*[int(x) for x in t_per_seq])
    _check(load().rswa_cache_set_t(handle, arr, _stream(stream)),
           "rswa_cache_set_t")


def rswa_cache_kv_offsets(handle):
    ko, vo = _c_size(0), _c_size(0)
    _check(load().rswa_cache_kv_offsets(handle, ctypes.byref(ko),
                                        ctypes.byref(vo)),
           "rswa_cache_kv_offsets")
    return ko.value, vo.value


def rswa_sync_status(handle) -> int:
    """Returns the status code (does not raise)."""
    return load().rswa_sync_status(handle)


class RswaCache:
    """A cache plus the torch-allocated device buffer that backs it."""

    def __init__(self, m, n, heads, head_dim, batch, dtype, device="cuda",
                 kv_heads=None):
        import torch
        self.m, self.n, self.heads, self.head_dim = m, n, heads, head_dim
        self.kv_heads = heads if kv_heads is None else kv_heads
        self.batch, self.dtype = batch, dtype
        nbytes = rswa_cache_footprint_gqa(m, n, heads, self.kv_heads, head_dim,
                                          batch, dtype)
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.handle = rswa_cache_create_gqa(m, n, heads, self.kv_heads,
                                            head_dim, batch, dtype, self.buf)

    def close(self):
        if self.handle is not None:
            rswa_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # thin forwards
    def prefill(self, Q, K, V, O, m_per_seq, T, stream=None):
        rswa_prefill(self.handle, Q, K, V, O, m_per_seq, T, stream)

    def prefill_varlen(self, Q, K, V, O, m_per_seq, t_per_seq, stream=None):
        rswa_prefill_varlen(self.handle, Q, K, V, O, m_per_seq, t_per_seq,
                            stream)

    def append_kv(self, k, v, stream=None):
        rswa_append_kv(self.handle, k, v, stream)

    def decode_step(self, q, o, lse=None, stream=None):
        rswa_decode_step(self.handle, q, o, lse, stream)

    def decode_step_fused(self, q, k, v, o, lse=None, stream=None):
        rswa_decode_step_fused(self.handle, q, k, v, o, lse, stream)

    def decode_block(self, q, k, v, o, lse=None, stream=None):
        rswa_decode_block(self.handle, q, k, v, o, lse, stream)

    def cache_bytes(self, b):
        return rswa_cache_bytes(self.handle, b)

    def cache_len(self, b):
        return rswa_cache_len(self.handle, b)

    def get_t(self, b):
        return rswa_cache_get_t(self.handle, b)

    def set_t(self, t_per_seq, stream=None):
        rswa_cache_set_t(self.handle, t_per_seq, stream)

    def sync_status(self):
        return rswa_sync_status(self.handle)

    def slabs(self):
        """(K, V) views of the cache slabs [B][H_kv][m + n][d] (for tests)."""
        import torch
        tdt = torch.float32 if self.dtype == RSWA_F32 else torch.bfloat16
        elt = 4 if self.dtype == RSWA_F32 else 2
        B, H, R, d = self.batch, self.kv_heads, self.m + self.n, self.head_dim
        nb = B * H * R * d * elt
        ko, vo = rswa_cache_kv_offsets(self.handle)
        Kt = self.buf[ko:ko + nb].view(tdt).view(B, H, R, d)
        Vt = self.buf[vo:vo + nb].view(tdt).view(B, H, R, d)
        return Kt, Vt
