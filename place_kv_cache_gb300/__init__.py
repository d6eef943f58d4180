"""Thin Python binding of the decode-step C ABI (``include/ol.h``).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of ``libol.so``. Functions keep the C names; they take torch tensors
(device memory), numpy arrays or plain integers for pointers, take the
caller's current CUDA stream by default, and raise ``OlError`` on any
non-OK status. There is no CPU fallback: if the library cannot be built or
loaded, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libol.so")

# ol_status
OL_OK, OL_ERR_NULL, OL_ERR_ALIAS, OL_ERR_READONLY, OL_ERR_CAPACITY, OL_ERR_SHAPE, OL_ERR_DTYPE, OL_ERR_BUSY, \
    OL_ERR_WORKSPACE, OL_ERR_CUDA, OL_ERR_UNSUPPORTED, OL_ERR_INJECTED, OL_ERR_PAGE, OL_ERR_ALIGN = range(14)
OL_F32, OL_BF16 = 0, 1
OL_READ_ONLY, OL_READ_WRITE = 0, 1
OL_HISTORY_STABLE = 0x100
OL_LAYOUT_CONTIGUOUS, OL_LAYOUT_PAGED, OL_LAYOUT_INT4, OL_LAYOUT_HPAGED = 0, 1, 2, 3
# ol_page_format_id: per-page element formats of the heterogeneous paged cache
OL_FMT_F32, OL_FMT_F16, OL_FMT_BF16, OL_FMT_I8, OL_FMT_U8, OL_FMT_I4, OL_FMT_U4, OL_FMT_I2, OL_FMT_U2 = range(9)
# host mirror of ol_page_format: (format, scale, zero point) of K, then of V
PAGE_FORMAT_DTYPE = np.dtype([("kf", "<i4"), ("ks", "<f4"), ("kz", "<i4"), ("vf", "<i4"), ("vs", "<f4"),
                              ("vz", "<i4")])
OL_Q_DYNAMIC, OL_Q_FIXED = 0, 1
OL_DEVICE_OK, OL_DEVICE_GUARD = 0, 1

SYMBOLS = ("ol_status_string", "ol_version", "ol_workspace_size", "ol_workspace_init", "ol_workspace_status",
           "ol_cache_bind", "ol_cache_unbind", "ol_cache_update", "ol_cache_update_rows",
           "ol_paged_cache_update", "ol_decode_attention", "ol_paged_decode_attention", "ol_int4kv_append",
           "ol_int4kv_decode_attention", "ol_decode_step", "ol_decode_step_noalloc", "ol_noalloc_status", "ol_workspace_size_host",
           "ol_decode_step_host", "ol_last_call_stats", "ol_total_stats", "ol_reset_stats",
           "ol_workspace_size_chunk", "ol_chunk_step", "ol_hpaged_append", "ol_hpaged_decode_attention",
           "ol_hpaged_decode_step", "ol_hpaged_quantize", "ol_hpaged_chunk_step")


class Stats(ctypes.Structure):
    """ol_stats: storage statistics of a call (see include/ol.h)."""
    _fields_ = [(n, ctypes.c_int64) for n in (
        "calls", "storage_allocations", "storage_allocated_bytes", "storage_prefix_copied_bytes",
        "storage_append_copied_bytes", "storage_reuse_count", "dequantized_bytes", "attended_tokens",
        "kv_payload_bytes_read", "workspace_bytes")]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


class OlError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_status_string(status)}")


class KVCache(ctypes.Structure):
    """ol_kv_cache: contiguous [2, batch, kv_heads, capacity, head_dim]."""
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("capacity", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("access", ctypes.c_int32), ("owner", ctypes.c_uint64)]


class PagedKV(ctypes.Structure):
    """ol_paged_kv: pool [2, num_pages, kv_heads, page_size, head_dim] + block table [batch, max_pages]."""
    _fields_ = [("data", ctypes.c_void_p), ("block_table", ctypes.c_void_p), ("block_table_host", ctypes.c_void_p),
                ("dtype", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("max_pages", ctypes.c_int32), ("access", ctypes.c_int32), ("owner", ctypes.c_uint64)]


class Int4KV(ctypes.Structure):
    """ol_int4_kv: codes / fp16 scales / zero-point planes of a [2, batch, kv_heads, capacity, head_dim] cache."""
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("zps", ctypes.c_void_p),
                ("batch", ctypes.c_int32), ("kv_heads", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("quant_mode", ctypes.c_int32), ("fixed_scale", ctypes.c_float),
                ("fixed_zp", ctypes.c_int32), ("access", ctypes.c_int32), ("owner", ctypes.c_uint64)]


class PlaneFormat(ctypes.Structure):
    """ol_plane_format: element format of one plane (K or V) of a page."""
    _fields_ = [("format", ctypes.c_int32), ("scale", ctypes.c_float), ("zero_point", ctypes.c_int32)]


class PageFormat(ctypes.Structure):
    """ol_page_format: the K and V formats of a page."""
    _fields_ = [("k", PlaneFormat), ("v", PlaneFormat)]


class HPagedKV(ctypes.Structure):
    """ol_hpaged_kv: page slots of 2 * kv_heads * page_size * head_dim * 4 bytes, per-page formats, block table."""
    _fields_ = [("pool", ctypes.c_void_p), ("formats", ctypes.c_void_p), ("formats_host", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("block_table_host", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("kv_heads", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("batch", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("access", ctypes.c_int32), ("owner", ctypes.c_uint64)]


_lib = None


def load(build_if_missing: bool = True, variant: str = ""):
    """Load libol.so (building it in-tree first if it is missing or stale).
    variant="phase" loads the timing build libol_phase.so instead (same API plus
    ol_debug_phase_stamps); it must be the first load of the process."""
    global _lib
    if _lib is not None:
        if variant and getattr(_lib, "_variant", "") != variant:
            raise RuntimeError(f"library already loaded without variant {variant!r}")
        return _lib
    path = LIB_PATH if not variant else os.path.join(_HERE, f"libol_{variant}.so")
    if build_if_missing:
        from . import _build
        try:
            _build.build(variant=variant)
        except Exception as e:  # no nvcc, compile error: fail loudly, never fall back
            if not os.path.exists(path):
                raise RuntimeError(f"the CUDA library could not be built: {e}") from e
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    L._variant = variant
    vp, i32, i64, u64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float,
                                  ctypes.c_size_t)
    st = ctypes.c_int
    sig = {
        "ol_status_string": (ctypes.c_char_p, [st]),
        "ol_version": (i32, []),
        "ol_workspace_size": (sz, [i32, i32, i32, i32]),
        "ol_workspace_init": (st, [vp, sz, vp]),
        "ol_workspace_status": (st, [vp, ctypes.POINTER(i32), vp]),
        "ol_cache_bind": (st, [vp, sz, u64]),
        "ol_cache_unbind": (st, [vp, u64]),
        "ol_cache_update": (st, [ctypes.POINTER(KVCache), vp, vp, i32, i64, vp]),
        "ol_cache_update_rows": (st, [ctypes.POINTER(KVCache), vp, vp, i32, vp, vp, vp]),
        "ol_paged_cache_update": (st, [ctypes.POINTER(PagedKV), vp, vp, i32, vp, vp, vp]),
        "ol_decode_attention": (st, [ctypes.POINTER(KVCache), vp, i32, vp, vp, f32, i32, vp, i32, vp, sz, vp]),
        "ol_paged_decode_attention": (st, [ctypes.POINTER(PagedKV), vp, i32, vp, vp, f32, i32, vp, i32, vp, sz, vp]),
        "ol_int4kv_append": (st, [ctypes.POINTER(Int4KV), vp, vp, vp, vp, vp]),
        "ol_int4kv_decode_attention": (st, [ctypes.POINTER(Int4KV), vp, i32, vp, vp, vp, f32, i32, vp, i32, vp, sz,
                                            vp]),
        "ol_decode_step": (st, [i32, vp, vp, vp, i32, vp, vp, vp, f32, i32, vp, i32, vp, sz, vp]),
        "ol_decode_step_noalloc": (st, [i32, vp, vp, vp, i32, vp, vp, vp, f32, i32, vp, i32, vp]),
        "ol_noalloc_status": (st, [ctypes.POINTER(i32), vp]),
        "ol_workspace_size_host": (sz, [i32, i32, i32, i32]),
        "ol_workspace_size_chunk": (sz, [i32, i32, i32, i32, i32]),
        "ol_chunk_step": (st, [i32, vp, vp, vp, i32, i32, vp, vp, vp, f32, i32, vp, i32, vp, sz, vp]),
        "ol_last_call_stats": (st, [vp]),
        "ol_total_stats": (st, [vp]),
        "ol_reset_stats": (None, []),
        "ol_decode_step_host": (st, [i32, vp, vp, vp, i32, vp, vp, f32, i32, vp, i32, vp, sz, vp]),
        "ol_hpaged_append": (st, [ctypes.POINTER(HPagedKV), vp, vp, i32, vp, vp, ctypes.POINTER(PageFormat), vp]),
        "ol_hpaged_decode_attention": (st, [ctypes.POINTER(HPagedKV), vp, i32, vp, vp, vp, f32, i32, vp, i32, vp, sz,
                                            vp]),
        "ol_hpaged_decode_step": (st, [ctypes.POINTER(HPagedKV), vp, vp, i32, vp, ctypes.POINTER(PageFormat), vp, vp,
                                       f32, i32, vp, i32, vp, sz, vp]),
        "ol_hpaged_quantize": (st, [ctypes.POINTER(HPagedKV), vp, vp, vp, vp, vp, i32, ctypes.POINTER(PageFormat),
                                    vp]),
        "ol_hpaged_chunk_step": (st, [ctypes.POINTER(HPagedKV), vp, vp, i32, i32, vp, ctypes.POINTER(PageFormat), vp,
                                      vp, f32, i32, vp, i32, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _status_string(s: int) -> str:
    try:
        return load(build_if_missing=False).ol_status_string(s).decode()
    except Exception:
        return f"status {s}"


# address getter per tensor type seen (torch.Tensor and subclasses): one dict
# lookup instead of the generic checks on every call of a per-step function
_PTR_OF_TYPE = {}
_I32 = np.dtype(np.int32)
_TORCH_I32 = None  # torch.int32, once torch is in use


def _ptr(x) -> Optional[int]:
    """Address of a torch tensor / numpy array / int (None stays NULL)."""
    get = _PTR_OF_TYPE.get(type(x))
    if get is not None:
        return get(x)
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    if hasattr(x, "data_ptr"):
        _PTR_OF_TYPE[type(x)] = type(x).data_ptr
        return x.data_ptr()
    raise TypeError(f"cannot take the address of {type(x)}")


def _host_i32(a):
    """Host int32 C-contiguous lengths/positions: the argument itself when it
    already is one (numpy array or CPU tensor), else a converted copy."""
    if a is None:
        return None
    global _TORCH_I32
    if type(a) is np.ndarray:
        if a.dtype == _I32 and a.flags.c_contiguous:
            return a
    elif type(a) in _PTR_OF_TYPE or hasattr(a, "data_ptr"):
        if _TORCH_I32 is None:
            import torch
            _TORCH_I32 = torch.int32
        if not a.is_cuda and a.dtype is _TORCH_I32 and a.is_contiguous():
            return a
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _stream(stream) -> Optional[int]:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except Exception:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != OL_OK:
        raise OlError(status, what)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return OL_BF16
    if t.dtype == torch.float32:
        return OL_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


# ------------------------------------------------------------- descriptors

def kv_cache(data, *, access: int = OL_READ_WRITE, owner: int = 0, dims=None, dtype: Optional[int] = None) -> KVCache:
    """Descriptor of a contiguous cache tensor [2, B, Hkv, C, D] (or a raw pointer with ``dims``)."""
    if dims is None:
        _, B, H, C, D = data.shape
        dtype = _dtype_code(data) if dtype is None else dtype
    else:
        B, H, C, D = dims
    d = KVCache(_ptr(data), dtype, B, H, C, D, access, owner)
    d._refs = (data,)  # the descriptor keeps the buffers it points to alive
    return d


def paged_kv(pool, block_table, block_table_host, *, access: int = OL_READ_WRITE, owner: int = 0, dims=None,
             dtype: Optional[int] = None) -> PagedKV:
    """Descriptor of a paged pool [2, P, Hkv, S, D] with a device and a host block table [B, M]."""
    bt_host = _host_i32(block_table_host)
    if dims is None:
        _, P, H, S, D = pool.shape
        dtype = _dtype_code(pool) if dtype is None else dtype
    else:
        P, H, S, D = dims
    B, M = bt_host.shape
    d = PagedKV(_ptr(pool), _ptr(block_table), _ptr(bt_host), dtype, P, H, S, D, B, M, access, owner)
    d._refs = (pool, block_table, bt_host)  # the descriptor keeps the buffers it points to alive
    return d


def int4_kv(codes, scales, zps, *, head_dim: Optional[int] = None, quant_mode: int = OL_Q_DYNAMIC,
            fixed_scale: float = 0.25, fixed_zp: int = 8, access: int = OL_READ_WRITE, owner: int = 0,
            dims=None) -> Int4KV:
    """Descriptor of INT4 planes: codes [2,B,H,C,D/2] u8, scales [2,B,H,C,D/32] fp16, zps [2,B,H,C,D/64] u8."""
    if dims is None:
        _, B, H, C, half = codes.shape
        D = half * 2 if head_dim is None else head_dim
    else:
        B, H, C, D = dims
    d = Int4KV(_ptr(codes), _ptr(scales), _ptr(zps), B, H, C, D, quant_mode, fixed_scale, fixed_zp, access, owner)
    d._refs = (codes, scales, zps)  # the descriptor keeps the buffers it points to alive
    return d


def page_format(k=(OL_FMT_BF16, 1.0, 0), v=(OL_FMT_BF16, 1.0, 0)) -> PageFormat:
    """A page's formats: k and v are (format, scale, zero point)."""
    return PageFormat(PlaneFormat(*k), PlaneFormat(*v))


def hpaged_kv(pool, formats, formats_host, block_table, block_table_host, *, kv_heads: int, page_size: int,
              head_dim: int, access: int = OL_READ_WRITE, owner: int = 0) -> HPagedKV:
    """Descriptor of a heterogeneous paged cache.

    pool: device bytes, num_pages slots of 2 * kv_heads * page_size * head_dim * 4;
    formats: device table of num_pages ol_page_format (24 bytes each);
    formats_host: the host mirror, a C-contiguous numpy array of PAGE_FORMAT_DTYPE
    that the library updates in place when a call starts or converts a page;
    block_table / block_table_host: [batch, max_pages] int32 on device / host.
    """
    if not (isinstance(formats_host, np.ndarray) and formats_host.dtype == PAGE_FORMAT_DTYPE
            and formats_host.flags.c_contiguous):
        raise TypeError("formats_host must be a C-contiguous numpy array of PAGE_FORMAT_DTYPE")
    bt_host = _host_i32(block_table_host)
    B, M = bt_host.shape
    P = formats_host.shape[0]
    d = HPagedKV(_ptr(pool), _ptr(formats), _ptr(formats_host), _ptr(block_table), _ptr(bt_host), P, kv_heads,
                 page_size, head_dim, B, M, access, owner)
    d._refs = (pool, formats, formats_host, block_table, bt_host)  # keeps the buffers alive
    return d


# ------------------------------------------------------------------ calls

def ol_version() -> int:
    return load().ol_version()


def ol_last_call_stats() -> dict:
    """Storage statistics of the last call on this thread that passed validation."""
    st = Stats()
    _check(load().ol_last_call_stats(ctypes.byref(st)), "ol_last_call_stats")
    return st.as_dict()


def ol_total_stats() -> dict:
    """Sums of the statistics of this thread's calls since ol_reset_stats."""
    st = Stats()
    _check(load().ol_total_stats(ctypes.byref(st)), "ol_total_stats")
    return st.as_dict()


def ol_reset_stats() -> None:
    load().ol_reset_stats()


def ol_status_string(status: int) -> str:
    return load().ol_status_string(status).decode()


def ol_workspace_size(batch: int, q_heads: int, kv_heads: int, head_dim: int) -> int:
    return load().ol_workspace_size(batch, q_heads, kv_heads, head_dim)


def ol_workspace_init(workspace, nbytes: Optional[int] = None, stream=None):
    nbytes = workspace.numel() * workspace.element_size() if nbytes is None else nbytes
    _check(load().ol_workspace_init(_ptr(workspace), nbytes, _stream(stream)), "ol_workspace_init")


def ol_workspace_status(workspace, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check(load().ol_workspace_status(_ptr(workspace), ctypes.byref(out), _stream(stream)), "ol_workspace_status")
    return out.value


def ol_cache_bind(base, nbytes: int, owner: int):
    _check(load().ol_cache_bind(_ptr(base), nbytes, owner), "ol_cache_bind")


def ol_cache_unbind(base, owner: int):
    _check(load().ol_cache_unbind(_ptr(base), owner), "ol_cache_unbind")


def ol_cache_update(cache: KVCache, updated, values, new_len: int, position: int, stream=None):
    _check(load().ol_cache_update(ctypes.byref(cache), _ptr(updated), _ptr(values), new_len, position,
                                  _stream(stream)), "ol_cache_update")


def ol_cache_update_rows(cache: KVCache, updated, values, new_len: int, positions_host, positions_dev, stream=None):
    ph = _host_i32(positions_host)
    _check(load().ol_cache_update_rows(ctypes.byref(cache), _ptr(updated), _ptr(values), new_len, _ptr(ph),
                                       _ptr(positions_dev), _stream(stream)), "ol_cache_update_rows")


def ol_paged_cache_update(kv: PagedKV, updated, values, new_len: int, positions_host, positions_dev, stream=None):
    ph = _host_i32(positions_host)
    _check(load().ol_paged_cache_update(ctypes.byref(kv), _ptr(updated), _ptr(values), new_len, _ptr(ph),
                                        _ptr(positions_dev), _stream(stream)), "ol_paged_cache_update")


def ol_decode_attention(cache: KVCache, q, q_heads: int, lens_host, lens_dev, scale: float, window: int, out,
                        out_dtype: int, workspace, ws_bytes: int, stream=None):
    lh = _host_i32(lens_host)
    _check(load().ol_decode_attention(ctypes.byref(cache), _ptr(q), q_heads, _ptr(lh), _ptr(lens_dev), scale, window,
                                      _ptr(out), out_dtype, _ptr(workspace), ws_bytes, _stream(stream)),
           "ol_decode_attention")


def ol_paged_decode_attention(kv: PagedKV, q, q_heads: int, lens_host, lens_dev, scale: float, window: int, out,
                              out_dtype: int, workspace, ws_bytes: int, stream=None):
    lh = _host_i32(lens_host)
    _check(load().ol_paged_decode_attention(ctypes.byref(kv), _ptr(q), q_heads, _ptr(lh), _ptr(lens_dev), scale,
                                            window, _ptr(out), out_dtype, _ptr(workspace), ws_bytes,
                                            _stream(stream)), "ol_paged_decode_attention")


def ol_int4kv_append(cache: Int4KV, updated_codes, values_bf16, positions_host, positions_dev, stream=None):
    ph = _host_i32(positions_host)
    _check(load().ol_int4kv_append(ctypes.byref(cache), _ptr(updated_codes), _ptr(values_bf16), _ptr(ph),
                                   _ptr(positions_dev), _stream(stream)), "ol_int4kv_append")


def ol_int4kv_decode_attention(cache: Int4KV, q, q_heads: int, lens_host, lens_dev, cur_kv, scale: float, window: int,
                               out, out_dtype: int, workspace, ws_bytes: int, stream=None):
    lh = _host_i32(lens_host)
    _check(load().ol_int4kv_decode_attention(ctypes.byref(cache), _ptr(q), q_heads, _ptr(lh), _ptr(lens_dev),
                                             _ptr(cur_kv), scale, window, _ptr(out), out_dtype, _ptr(workspace),
                                             ws_bytes, _stream(stream)), "ol_int4kv_decode_attention")


def ol_decode_step(layout: int, desc, updated, q, q_heads: int, new_kv, lens_host, lens_dev, scale: float,
                   window: int, out, out_dtype: int, workspace, ws_bytes: int, stream=None):
    lh = _host_i32(lens_host)
    _check(load().ol_decode_step(layout, ctypes.byref(desc), _ptr(updated), _ptr(q), q_heads, _ptr(new_kv), _ptr(lh),
                                 _ptr(lens_dev), scale, window, _ptr(out), out_dtype, _ptr(workspace), ws_bytes,
                                 _stream(stream)), "ol_decode_step")


def ol_workspace_size_chunk(batch: int, q_heads: int, kv_heads: int, head_dim: int, new_len: int) -> int:
    return load().ol_workspace_size_chunk(batch, q_heads, kv_heads, head_dim, new_len)


def ol_chunk_step(layout: int, desc, updated, q, q_heads: int, new_len: int, new_kv, lens_host, lens_dev,
                  scale: float, window: int, out, out_dtype: int, workspace, ws_bytes: int, stream=None):
    """Append new_len tokens per row and attend causally inside the chunk:
    q and out [B, Hq, new_len, D], new_kv [2, B, Hkv, new_len, D]."""
    lh = _host_i32(lens_host)
    _check(load().ol_chunk_step(layout, ctypes.byref(desc), _ptr(updated), _ptr(q), q_heads, new_len, _ptr(new_kv),
                                _ptr(lh), _ptr(lens_dev), scale, window, _ptr(out), out_dtype, _ptr(workspace),
                                ws_bytes, _stream(stream)), "ol_chunk_step")


def ol_workspace_size_host(batch: int, q_heads: int, kv_heads: int, head_dim: int) -> int:
    return load().ol_workspace_size_host(batch, q_heads, kv_heads, head_dim)


def ol_decode_step_host(layout: int, desc, updated, q_host, q_heads: int, new_kv_host, lens_host, scale: float,
                        window: int, out_host, out_dtype: int, workspace, ws_bytes: int, stream=None):
    """ol_decode_step with q, new K/V, lengths and y in host memory (numpy arrays
    or CPU tensors, pinned for asynchronous copies); y is in out_host once the
    stream has been synchronized."""
    lh = _host_i32(lens_host)
    _check(load().ol_decode_step_host(layout, ctypes.byref(desc), _ptr(updated), _ptr(q_host), q_heads,
                                      _ptr(new_kv_host), _ptr(lh), scale, window, _ptr(out_host), out_dtype,
                                      _ptr(workspace), ws_bytes, _stream(stream)), "ol_decode_step_host")


def ol_decode_step_noalloc(layout: int, desc, updated, q, q_heads: int, new_kv, lens_host, lens_dev, scale: float,
                           window: int, out, out_dtype: int, stream=None):
    """ol_decode_step without a workspace argument, for callers that cannot
    allocate: the library's own static device scratch serves as workspace."""
    lh = _host_i32(lens_host)
    _check(load().ol_decode_step_noalloc(layout, ctypes.byref(desc), _ptr(updated), _ptr(q), q_heads, _ptr(new_kv),
                                         _ptr(lh), _ptr(lens_dev), scale, window, _ptr(out), out_dtype,
                                         _stream(stream)), "ol_decode_step_noalloc")


def ol_noalloc_status(stream=None) -> int:
    """Read and clear the status word of the allocation-free step's scratch (current device)."""
    out = ctypes.c_int32(0)
    _check(load().ol_noalloc_status(ctypes.byref(out), _stream(stream)), "ol_noalloc_status")
    return out.value


def ol_hpaged_append(kv: HPagedKV, updated, values, new_len: int, positions_host, positions_dev,
                     new_pages: PageFormat, stream=None):
    """values [2, B, Hkv, new_len, D] bf16 at positions[b]; pages the append starts take new_pages."""
    ph = _host_i32(positions_host)
    _check(load().ol_hpaged_append(ctypes.byref(kv), _ptr(updated), _ptr(values), new_len, _ptr(ph),
                                   _ptr(positions_dev), ctypes.byref(new_pages), _stream(stream)), "ol_hpaged_append")


def ol_hpaged_decode_attention(kv: HPagedKV, q, q_heads: int, lens_host, lens_dev, cur_kv, scale: float, window: int,
                               out, out_dtype: int, workspace, ws_bytes: int, stream=None):
    lh = _host_i32(lens_host)
    _check(load().ol_hpaged_decode_attention(ctypes.byref(kv), _ptr(q), q_heads, _ptr(lh), _ptr(lens_dev),
                                             _ptr(cur_kv), scale, window, _ptr(out), out_dtype, _ptr(workspace),
                                             ws_bytes, _stream(stream)), "ol_hpaged_decode_attention")


def ol_hpaged_decode_step(kv: HPagedKV, updated, q, q_heads: int, new_kv, new_pages: PageFormat, lens_host, lens_dev,
                          scale: float, window: int, out, out_dtype: int, workspace, ws_bytes: int, stream=None):
    lh = _host_i32(lens_host)
    _check(load().ol_hpaged_decode_step(ctypes.byref(kv), _ptr(updated), _ptr(q), q_heads, _ptr(new_kv),
                                        ctypes.byref(new_pages), _ptr(lh), _ptr(lens_dev), scale, window, _ptr(out),
                                        out_dtype, _ptr(workspace), ws_bytes, _stream(stream)),
           "ol_hpaged_decode_step")


def ol_hpaged_quantize(kv: HPagedKV, updated, pages_host, pages_dev, valid_host, valid_dev, to: PageFormat,
                       stream=None):
    """QuantizePagedCache on the selected pages: valid prefixes converted to `to`, the rest zero."""
    ph, vh = _host_i32(pages_host), _host_i32(valid_host)
    _check(load().ol_hpaged_quantize(ctypes.byref(kv), _ptr(updated), _ptr(ph), _ptr(pages_dev), _ptr(vh),
                                     _ptr(valid_dev), len(ph), ctypes.byref(to), _stream(stream)),
           "ol_hpaged_quantize")


def ol_hpaged_chunk_step(kv: HPagedKV, updated, q, q_heads: int, new_len: int, new_kv, new_pages: PageFormat,
                         lens_host, lens_dev, scale: float, window: int, out, out_dtype: int, workspace,
                         ws_bytes: int, stream=None):
    """Chunked step on heterogeneous pages: q and out [B, Hq, new_len, D], new_kv [2, B, Hkv, new_len, D]."""
    lh = _host_i32(lens_host)
    _check(load().ol_hpaged_chunk_step(ctypes.byref(kv), _ptr(updated), _ptr(q), q_heads, new_len, _ptr(new_kv),
                                       ctypes.byref(new_pages), _ptr(lh), _ptr(lens_dev), scale, window, _ptr(out),
                                       out_dtype, _ptr(workspace), ws_bytes, _stream(stream)), "ol_hpaged_chunk_step")
