"""Python access to the CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: this package is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``; the
product path (``place_kv_cache_gb300``) never imports, loads or calls it, and
the two share no code.

Arrays are numpy: bf16 values are ``uint16`` bit patterns, fp32 values are
``float32``. Attention results are fp64. Every wrapper returns the oracle's
result or raises ``OracleError`` with the oracle's status code.

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, invariants and the figures printed on the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# gcc command that builds the oracle; __graft_entry__.build() runs the same line.
BUILD_CMD = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
             "-o", _LIB, _SRC, "-lm"]

F32, BF16 = 0, 1
Q_DYNAMIC, Q_FIXED = 0, 1


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.run(BUILD_CMD, check=True)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp, i32, f64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_float
        L.orc_visible_range.argtypes = [i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        L.orc_decode_attention.argtypes = [vp, i32, i32, vp, i32, i32, i32, i32, i32, vp, f64, i32, vp]
        L.orc_paged_attention.argtypes = [vp, i32, i32, vp, i32, i32, i32, i32, i32, vp, i32, i32, vp,
                                          f64, i32, vp]
        L.orc_cache_update.argtypes = [vp, i32, i32, i32, i32, i32, vp, i32, vp]
        L.orc_paged_update.argtypes = [vp, i32, i32, i32, i32, i32, vp, i32, i32, vp, i32, vp]
        L.orc_pack_u4.argtypes = [vp, i32, vp]
        L.orc_pack_u4.restype = None
        L.orc_unpack_u4.argtypes = [vp, i32, vp]
        L.orc_unpack_u4.restype = None
        L.orc_int4_quantize_row.argtypes = [vp, i32, i32, f32, i32, vp, vp, vp]
        L.orc_int4_dequantize_row.argtypes = [vp, vp, vp, i32, vp]
        L.orc_int4_append.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, i32, vp, i32, f32, i32]
        L.orc_int4_attention.argtypes = [vp, i32, vp, vp, vp, i32, i32, i32, i32, vp, vp, f64, i32, vp]
        L.orc_fp16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_fp16_to_double.restype = f64
        L.orc_float_to_fp16.argtypes = [f32]
        L.orc_float_to_fp16.restype = ctypes.c_uint16
        L.orc_hf_encode_row.argtypes = [vp, i32, vp, vp]
        L.orc_hf_decode_row.argtypes = [vp, i32, vp, vp]
        L.orc_hpaged_append.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, i32, vp, i32, vp, vp]
        L.orc_hpaged_attention.argtypes = [vp, i32, vp, vp, i32, i32, i32, i32, vp, i32, i32, vp, vp, f64, i32, vp]
        L.orc_hpaged_quantize.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, i32, vp]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what}: oracle status {rc}")


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes float32 or uint16 (bf16 bits), got {a.dtype}")


def _c(a, dtype=None):
    return np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype=dtype))


def default_scale(head_dim: int) -> float:
    return 1.0 / float(np.sqrt(head_dim))


def visible_range(n: int, window: int = -1):
    lo, hi = ctypes.c_int(), ctypes.c_int()
    lib().orc_visible_range(n, window, ctypes.byref(lo), ctypes.byref(hi))
    return lo.value, hi.value


def decode_attention(q, cache, lens, scale: Optional[float] = None, window: int = -1) -> np.ndarray:
    """q [B, Hq, D]; cache [2, B, Hkv, C, D]; lens [B] -> y [B, Hq, D] fp64."""
    q, cache, lens = _c(q), _c(cache), _c(lens, np.int32)
    B, Hq, D = q.shape
    _, B2, Hkv, C, D2 = cache.shape
    assert B == B2 and D == D2
    out = np.zeros((B, Hq, D), dtype=np.float64)
    s = default_scale(D) if scale is None else scale
    _check(lib().orc_decode_attention(_ptr(q), _dtype_code(q), Hq, _ptr(cache), _dtype_code(cache),
                                      B, Hkv, C, D, _ptr(lens), s, window, _ptr(out)), "decode_attention")
    return out


def paged_attention(q, pool, block_table, lens, scale: Optional[float] = None, window: int = -1) -> np.ndarray:
    """q [B, Hq, D]; pool [2, P, Hkv, S, D]; block_table [B, M] -> y [B, Hq, D] fp64."""
    q, pool, bt, lens = _c(q), _c(pool), _c(block_table, np.int32), _c(lens, np.int32)
    B, Hq, D = q.shape
    _, P, Hkv, S, D2 = pool.shape
    assert D == D2 and bt.shape[0] == B
    out = np.zeros((B, Hq, D), dtype=np.float64)
    s = default_scale(D) if scale is None else scale
    _check(lib().orc_paged_attention(_ptr(q), _dtype_code(q), Hq, _ptr(pool), _dtype_code(pool), P, Hkv, S,
                                     D, _ptr(bt), bt.shape[1], B, _ptr(lens), s, window, _ptr(out)),
           "paged_attention")
    return out


def chunk_attention(q, cache, lens, new_len: int, scale: Optional[float] = None, window: int = -1) -> np.ndarray:
    """Causal attention inside a chunk of new_len appended tokens (the Attention
    contract of page "Persistent input/output feedback", section Optional
    heterogeneous paged KV: causal masking by default, left window). Query
    token i of row b sits at position p_i = lens[b] - new_len + i and attends
    the visible range of that position, which is exactly a decode attention
    over a prefix of p_i + 1 tokens. q [B, Hq, new_len, D]; the cache already
    holds the appended tokens -> y [B, Hq, new_len, D] fp64."""
    lens = _c(lens, np.int32)
    return np.stack([decode_attention(np.ascontiguousarray(q[:, :, i, :]), cache, lens - new_len + i + 1,
                                      scale=scale, window=window) for i in range(new_len)], axis=2)


def paged_chunk_attention(q, pool, block_table, lens, new_len: int, scale: Optional[float] = None,
                          window: int = -1) -> np.ndarray:
    """chunk_attention over a paged pool."""
    lens = _c(lens, np.int32)
    return np.stack([paged_attention(np.ascontiguousarray(q[:, :, i, :]), pool, block_table,
                                     lens - new_len + i + 1, scale=scale, window=window)
                     for i in range(new_len)], axis=2)


def cache_update(cache: np.ndarray, values, positions) -> None:
    """In place: cache [2, B, H, C, D]; values [2, B, H, new_len, D]; positions [B]."""
    assert cache.flags.c_contiguous
    values, positions = _c(values, cache.dtype), _c(positions, np.int32)
    _, B, H, C, D = cache.shape
    new_len = values.shape[3]
    assert values.shape == (2, B, H, new_len, D)
    _check(lib().orc_cache_update(_ptr(cache), _dtype_code(cache), B, H, C, D, _ptr(values), new_len,
                                  _ptr(positions)), "cache_update")


def paged_update(pool: np.ndarray, block_table, values, positions) -> None:
    """In place: pool [2, P, H, S, D]; block_table [B, M]; values [2, B, H, new_len, D]."""
    assert pool.flags.c_contiguous
    bt, values, positions = _c(block_table, np.int32), _c(values, pool.dtype), _c(positions, np.int32)
    _, P, H, S, D = pool.shape
    B, M = bt.shape
    new_len = values.shape[3]
    assert values.shape == (2, B, H, new_len, D)
    _check(lib().orc_paged_update(_ptr(pool), _dtype_code(pool), P, H, S, D, _ptr(bt), M, B, _ptr(values),
                                  new_len, _ptr(positions)), "paged_update")


def pack_u4(codes) -> np.ndarray:
    codes = _c(codes, np.uint8)
    out = np.zeros((codes.size + 1) // 2, dtype=np.uint8)
    lib().orc_pack_u4(_ptr(codes), codes.size, _ptr(out))
    return out


def unpack_u4(packed, n: int) -> np.ndarray:
    packed = _c(packed, np.uint8)
    out = np.zeros(n, dtype=np.uint8)
    lib().orc_unpack_u4(_ptr(packed), n, _ptr(out))
    return out


def int4_row_bytes(D: int):
    """(code bytes, scales, zero-point bytes) of one token row of one head."""
    return D // 2, D // 32, (D // 32 + 1) // 2


def int4_quantize_row(x_bf16, mode: int = Q_DYNAMIC, fixed_scale: float = 0.25, fixed_zp: int = 8):
    """One token's D bf16 values -> (codes [D/2] u8, scales [D/32] fp16 bits, zps [ceil(D/64)] u8)."""
    x = _c(x_bf16, np.uint16)
    D = x.size
    cb, sb, zb = int4_row_bytes(D)
    codes = np.zeros(cb, np.uint8)
    scales = np.zeros(sb, np.uint16)
    zps = np.zeros(zb, np.uint8)
    _check(lib().orc_int4_quantize_row(_ptr(x), D, mode, fixed_scale, fixed_zp, _ptr(codes), _ptr(scales),
                                       _ptr(zps)), "int4_quantize_row")
    return codes, scales, zps


def int4_dequantize_row(codes, scales, zps) -> np.ndarray:
    codes, scales, zps = _c(codes, np.uint8), _c(scales, np.uint16), _c(zps, np.uint8)
    D = codes.size * 2
    out = np.zeros(D, np.float64)
    _check(lib().orc_int4_dequantize_row(_ptr(codes), _ptr(scales), _ptr(zps), D, _ptr(out)),
           "int4_dequantize_row")
    return out


def int4_planes(B: int, H: int, C: int, D: int):
    """Fresh zeroed INT4 planes (codes, scales, zps) for a [2, B, H, C, D] logical cache."""
    cb, sb, zb = int4_row_bytes(D)
    return (np.zeros((2, B, H, C, cb), np.uint8), np.zeros((2, B, H, C, sb), np.uint16),
            np.zeros((2, B, H, C, zb), np.uint8))


def int4_append(codes, scales, zps, values_bf16, positions, mode: int = Q_DYNAMIC,
                fixed_scale: float = 0.25, fixed_zp: int = 8) -> None:
    """In place on the planes; values [2, B, H, new_len, D] bf16 bits."""
    for a in (codes, scales, zps):
        assert a.flags.c_contiguous
    values, positions = _c(values_bf16, np.uint16), _c(positions, np.int32)
    _, B, H, new_len, D = values.shape
    C = codes.shape[3]
    _check(lib().orc_int4_append(_ptr(codes), _ptr(scales), _ptr(zps), B, H, C, D, _ptr(values), new_len,
                                 _ptr(positions), mode, fixed_scale, fixed_zp), "int4_append")


def int4_attention(q, codes, scales, zps, lens, cur_kv=None, scale: Optional[float] = None,
                   window: int = -1) -> np.ndarray:
    """q [B, Hq, D] bf16 bits; planes as from int4_planes; cur_kv [2, B, Hkv, 1, D] bf16 or None."""
    q, codes, scales, zps, lens = _c(q, np.uint16), _c(codes), _c(scales), _c(zps), _c(lens, np.int32)
    B, Hq, D = q.shape
    _, B2, Hkv, C, _cb = codes.shape
    assert B == B2
    cur = None if cur_kv is None else _c(cur_kv, np.uint16)
    out = np.zeros((B, Hq, D), np.float64)
    s = default_scale(D) if scale is None else scale
    _check(lib().orc_int4_attention(_ptr(q), Hq, _ptr(codes), _ptr(scales), _ptr(zps), B, Hkv, C, D,
                                    _ptr(lens), _ptr(cur), s, window, _ptr(out)), "int4_attention")
    return out


def int4_chunk_attention(q, codes, scales, zps, lens, new_len: int, new_kv, scale: Optional[float] = None,
                         window: int = -1) -> np.ndarray:
    """Chunked step over the INT4 cache: query token i of row b sits at
    p_i = lens[b] - new_len + i and attends its causal, windowed range; the
    history [0, lens[b] - new_len) is read from the codes (decoded), the
    chunk's own tokens take part uncompressed from new_kv (page "Persistent
    input/output feedback", Optional heterogeneous paged KV: current K/V are
    attended as uncompressed values and encoded only afterwards).
    q [B, Hq, new_len, D] bf16 bits; new_kv [2, B, Hkv, new_len, D] bf16 bits
    -> y [B, Hq, new_len, D] fp64. Built as the pinned chunk_attention over a
    float32 cache holding exactly those values (each decoded value (c - zp) *
    scale is exact in float32)."""
    codes, scales, zps, lens = _c(codes), _c(scales), _c(zps), _c(lens, np.int32)
    new_kv = _c(new_kv, np.uint16)
    _, B, H, C, _cb = codes.shape
    D = new_kv.shape[4]
    dense = np.full((2, B, H, C, D), np.nan, np.float32)
    for b in range(B):
        hist = int(lens[b]) - new_len
        for plane in range(2):
            for h in range(H):
                for t in range(hist):
                    dense[plane, b, h, t] = int4_dequantize_row(codes[plane, b, h, t], scales[plane, b, h, t],
                                                                zps[plane, b, h, t])
                bits = new_kv[plane, b, h].astype(np.uint32) << 16
                dense[plane, b, h, hist:hist + new_len] = bits.view(np.float32)
    return chunk_attention(q, dense, lens, new_len, scale=scale, window=window)


def fp16_to_float(bits: int) -> float:
    return float(lib().orc_fp16_to_double(int(bits)))


def float_to_fp16(f: float) -> int:
    return int(lib().orc_float_to_fp16(float(f)))


# ------------------------------------------------ heterogeneous paged pages

# Page formats (the oracle's own numbering, which the library's enumeration
# mirrors): dense FLOAT, FLOAT16, BFLOAT16; affine INT8, UINT8, INT4, UINT4,
# INT2, UINT2.
HF_F32, HF_F16, HF_BF16, HF_I8, HF_U8, HF_I4, HF_U4, HF_I2, HF_U2 = range(9)
HF_BITS = {HF_F32: 32, HF_F16: 16, HF_BF16: 16, HF_I8: 8, HF_U8: 8, HF_I4: 4, HF_U4: 4, HF_I2: 2, HF_U2: 2}
HF_RANGE = {HF_I8: (-128, 127), HF_U8: (0, 255), HF_I4: (-8, 7), HF_U4: (0, 15), HF_I2: (-2, 1), HF_U2: (0, 3)}

# one page's descriptor: (format, scale, zero point) of K, then of V
PAGE_DESC = np.dtype([("kf", "<i4"), ("ks", "<f4"), ("kz", "<i4"), ("vf", "<i4"), ("vs", "<f4"), ("vz", "<i4")])


def page_desc(k=(HF_BF16, 1.0, 0), v=(HF_BF16, 1.0, 0)) -> np.ndarray:
    """A one-element descriptor array for K format k and V format v."""
    d = np.zeros(1, PAGE_DESC)
    d["kf"], d["ks"], d["kz"] = k
    d["vf"], d["vs"], d["vz"] = v
    return d


def hpaged_pool(P: int, H: int, S: int, D: int):
    """Zeroed page slots [P, 2 * H * S * D * 4] bytes and descriptors [P] (all BFLOAT16)."""
    desc = np.zeros(P, PAGE_DESC)
    desc["kf"] = HF_BF16
    desc["vf"] = HF_BF16
    return np.zeros((P, 2 * H * S * D * 4), np.uint8), desc


def hf_encode_row(x_bf16, fmt) -> np.ndarray:
    """Codes of one row of D bf16 values in plane format fmt = (format, scale, zp)."""
    x = _c(x_bf16, np.uint16)
    D = x.shape[0]
    out = np.zeros((D * HF_BITS[fmt[0]] + 7) // 8, np.uint8)
    f = page_desc(k=fmt)
    _check(lib().orc_hf_encode_row(_ptr(x), D, _ptr(f), _ptr(out)), "hf_encode_row")
    return out


def hf_decode_row(row, D: int, fmt) -> np.ndarray:
    """fp32 reconstructions (as fp64) of one row of D elements in format fmt."""
    r = _c(row, np.uint8)
    out = np.zeros(D, np.float64)
    f = page_desc(k=fmt)
    _check(lib().orc_hf_decode_row(_ptr(r), D, _ptr(f), _ptr(out)), "hf_decode_row")
    return out


def hpaged_append(pool, desc, block_table, values, positions, new_fmt) -> None:
    """In place: values [2, B, H, new_len, D] bf16 at positions [B]; new_fmt a
    one-element PAGE_DESC array for pages the append starts."""
    assert pool.flags.c_contiguous and desc.flags.c_contiguous
    bt, values, positions = _c(block_table, np.int32), _c(values, np.uint16), _c(positions, np.int32)
    _, B, H, new_len, D = values.shape
    P = pool.shape[0]
    S = pool.shape[1] // (2 * H * D * 4)
    _check(lib().orc_hpaged_append(_ptr(pool), _ptr(desc), P, H, S, D, _ptr(bt), bt.shape[1], B, _ptr(values),
                                   new_len, _ptr(positions), _ptr(_c(new_fmt, PAGE_DESC))), "hpaged_append")


def hpaged_attention(q, pool, desc, block_table, lens, H: int, cur_kv=None, scale: Optional[float] = None,
                     window: int = -1) -> np.ndarray:
    """q [B, Hq, D] bf16 over the heterogeneous pages (H kv heads) -> y fp64."""
    q, bt, lens = _c(q, np.uint16), _c(block_table, np.int32), _c(lens, np.int32)
    B, Hq, D = q.shape
    P = pool.shape[0]
    S = pool.shape[1] // (2 * H * D * 4)
    out = np.zeros((B, Hq, D), np.float64)
    s = default_scale(D) if scale is None else scale
    cur = None if cur_kv is None else _c(cur_kv, np.uint16)
    _check(lib().orc_hpaged_attention(_ptr(q), Hq, _ptr(_c(pool, np.uint8)), _ptr(_c(desc, PAGE_DESC)), P, H, S,
                                      D, _ptr(bt), bt.shape[1], B, _ptr(lens), _ptr(cur), s, window, _ptr(out)),
           "hpaged_attention")
    return out


def hpaged_chunk_attention(q, pool, desc, block_table, lens, H: int, new_len: int, new_kv,
                           scale: Optional[float] = None, window: int = -1) -> np.ndarray:
    """Chunked step over the heterogeneous pages: query token i of row b at
    p_i = lens[b] - new_len + i attends its causal, windowed range; history
    [0, lens[b] - new_len) decoded by each page's formats, the chunk's tokens
    uncompressed from new_kv (page "Persistent input/output feedback",
    Optional heterogeneous paged KV: current K/V attended uncompressed, encoded
    afterwards). q [B, Hq, new_len, D], new_kv [2, B, H, new_len, D] bf16 bits
    -> y [B, Hq, new_len, D] fp64: the pinned chunk_attention over a float32
    cache holding exactly those values (every decoded value is an fp32)."""
    bt, lens, new_kv = _c(block_table, np.int32), _c(lens, np.int32), _c(new_kv, np.uint16)
    B, M = bt.shape
    D = new_kv.shape[4]
    S = pool.shape[1] // (2 * H * D * 4)
    plane_bytes = H * S * D * 4
    dense = np.full((2, B, H, M * S, D), np.nan, np.float32)
    for b in range(B):
        hist = int(lens[b]) - new_len
        for t in range(hist):
            page, slot = int(bt[b, t // S]), t % S
            for plane, (f, sc, zp) in enumerate(((desc["kf"][page], desc["ks"][page], desc["kz"][page]),
                                                  (desc["vf"][page], desc["vs"][page], desc["vz"][page]))):
                rb = D * HF_BITS[int(f)] // 8
                for h in range(H):
                    off = plane * plane_bytes + (h * S + slot) * rb
                    dense[plane, b, h, t] = hf_decode_row(pool[page, off:off + rb], D, (int(f), float(sc), int(zp)))
        for plane in range(2):
            bits = new_kv[plane, b].astype(np.uint32) << 16
            dense[plane, b, :, hist:hist + new_len] = bits.view(np.float32)
    return chunk_attention(q, dense, lens, new_len, scale=scale, window=window)


def hpaged_quantize(pool, desc, H: int, D: int, pages, valid, to_fmt) -> None:
    """In place (QuantizePagedCache): the selected pages' valid prefixes converted
    to to_fmt (a one-element PAGE_DESC array), the rest zero in that format."""
    assert pool.flags.c_contiguous and desc.flags.c_contiguous
    pg, va = _c(pages, np.int32), _c(valid, np.int32)
    P = pool.shape[0]
    S = pool.shape[1] // (2 * H * D * 4)
    _check(lib().orc_hpaged_quantize(_ptr(pool), _ptr(desc), P, H, S, D, _ptr(pg), _ptr(va), pg.shape[0],
                                     _ptr(_c(to_fmt, PAGE_DESC))), "hpaged_quantize")
