"""CPU tests of the C ABI: the library loads, exports every symbol the header
declares, and rejects every invalid request on the host before any launch.

No GPU is touched: device pointers here are fake aligned addresses that host
validation compares but never dereferences. Valid requests are stopped right
after validation by the host fault-injection switch (OL_FAULT_INJECT), so they
never reach the CUDA runtime.
"""
import os
import re

import numpy as np
import pytest

import place_kv_cache_gb300 as ol

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ol.h")

BASE = 0x7F0000000000     # fake device address space, 16-byte aligned
MB = 1 << 20


@pytest.fixture(autouse=True)
def _inject(monkeypatch):
    monkeypatch.setenv("OL_FAULT_INJECT", "after_validate")
    yield


def header_symbols():
    with open(HEADER) as f:
        return re.findall(r"^OL_API [^(]*?\b(ol_\w+)\(", f.read(), flags=re.M)


def test_library_exports_every_declared_symbol():
    lib = ol.load()
    names = header_symbols()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(ol.SYMBOLS)
    assert ol.ol_version() == 100


def test_status_strings_cover_every_code():
    for code in range(14):
        s = ol.ol_status_string(code)
        assert s.startswith("OL_OK" if code == 0 else "OL_ERR_")


def test_workspace_size_grows_with_batch():
    a = ol.ol_workspace_size(1, 32, 8, 128)
    b = ol.ol_workspace_size(32, 32, 8, 128)
    assert a > 0 and b > a
    assert ol.ol_workspace_size(1, 7, 4, 128) == 0     # q_heads not a multiple of kv_heads


# ---------------------------------------------------------------- helpers

B, HQ, HKV, C, D = 2, 8, 2, 64, 128
CACHE = BASE
CACHE_BYTES = 2 * B * HKV * C * D * 2
Q = BASE + 64 * MB
NEWKV = BASE + 65 * MB
OUT = BASE + 66 * MB
LENS_DEV = BASE + 67 * MB
WS = BASE + 68 * MB
WS_BYTES = ol.ol_workspace_size(B, HQ, HKV, D)


def step(desc=None, updated=CACHE, q=Q, new_kv=NEWKV, lens=(10, 64), out=OUT, ws=WS, ws_bytes=WS_BYTES,
         q_heads=HQ, layout=ol.OL_LAYOUT_CONTIGUOUS):
    desc = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16) if desc is None else desc
    ol.ol_decode_step(layout, desc, updated, q, q_heads, new_kv, np.array(lens, np.int32), LENS_DEV, 0.0, -1, out,
                      ol.OL_BF16, ws, ws_bytes, stream=0)


def status_of(fn, *a, **k):
    try:
        fn(*a, **k)
    except ol.OlError as e:
        return e.status
    return ol.OL_OK


# ------------------------------------------------------------ contiguous


def test_valid_step_passes_validation():
    assert status_of(step) == ol.OL_ERR_INJECTED


def test_pointer_identity_is_required():
    assert status_of(step, updated=CACHE + 256) == ol.OL_ERR_ALIAS
    assert status_of(step, updated=None) == ol.OL_ERR_NULL


def test_read_only_cache_is_rejected():
    desc = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16, access=ol.OL_READ_ONLY)
    assert status_of(step, desc=desc) == ol.OL_ERR_READONLY


def test_capacity_is_checked_never_grown():
    assert status_of(step, lens=(10, 65)) == ol.OL_ERR_CAPACITY     # append at 64 == capacity
    assert status_of(step, lens=(0, 5)) == ol.OL_ERR_CAPACITY       # a step needs lens >= 1
    assert status_of(step, lens=(-1, 5)) == ol.OL_ERR_CAPACITY


def test_buffers_overlapping_the_cache_are_rejected():
    assert status_of(step, q=CACHE + 4096) == ol.OL_ERR_ALIAS
    assert status_of(step, new_kv=CACHE + CACHE_BYTES - 16) == ol.OL_ERR_ALIAS
    assert status_of(step, out=CACHE) == ol.OL_ERR_ALIAS
    assert status_of(step, ws=CACHE + 1024) == ol.OL_ERR_ALIAS
    assert status_of(step, q=CACHE + CACHE_BYTES) == ol.OL_ERR_INJECTED   # adjacent, not overlapping
    assert status_of(step, out=Q) == ol.OL_ERR_ALIAS                      # output over an input


def test_workspace_and_alignment_and_shape():
    assert status_of(step, ws_bytes=WS_BYTES - 1) == ol.OL_ERR_WORKSPACE
    assert status_of(step, ws=None) == ol.OL_ERR_NULL
    assert status_of(step, q=Q + 8) == ol.OL_ERR_ALIGN
    assert status_of(step, q_heads=7) == ol.OL_ERR_SHAPE
    desc = ol.kv_cache(CACHE + 8, dims=(B, HKV, C, D), dtype=ol.OL_BF16)
    assert status_of(step, desc=desc, updated=CACHE + 8) == ol.OL_ERR_ALIGN
    desc = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=7)
    assert status_of(step, desc=desc) == ol.OL_ERR_DTYPE


def test_cache_update_scalar_position():
    desc = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16)
    assert status_of(ol.ol_cache_update, desc, CACHE, NEWKV, 1, 63, stream=0) == ol.OL_ERR_INJECTED
    assert status_of(ol.ol_cache_update, desc, CACHE, NEWKV, 2, 63, stream=0) == ol.OL_ERR_CAPACITY
    assert status_of(ol.ol_cache_update, desc, CACHE, NEWKV, 1, -1, stream=0) == ol.OL_ERR_CAPACITY
    assert status_of(ol.ol_cache_update, desc, CACHE + 16, NEWKV, 1, 0, stream=0) == ol.OL_ERR_ALIAS
    assert status_of(ol.ol_cache_update, desc, CACHE, CACHE + 32, 1, 0, stream=0) == ol.OL_ERR_ALIAS


def test_cache_update_rows_positions():
    desc = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16)
    ok = status_of(ol.ol_cache_update_rows, desc, CACHE, NEWKV, 4, [0, 60], LENS_DEV, stream=0)
    assert ok == ol.OL_ERR_INJECTED
    bad = status_of(ol.ol_cache_update_rows, desc, CACHE, NEWKV, 4, [0, 61], LENS_DEV, stream=0)
    assert bad == ol.OL_ERR_CAPACITY


def test_attention_needs_no_write_access():
    desc = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16, access=ol.OL_READ_ONLY)
    s = status_of(ol.ol_decode_attention, desc, Q, HQ, [0, 64], LENS_DEV, 0.0, -1, OUT, ol.OL_F32, WS, WS_BYTES,
                  stream=0)
    assert s == ol.OL_ERR_INJECTED
    s = status_of(ol.ol_decode_attention, desc, Q, HQ, [0, 65], LENS_DEV, 0.0, -1, OUT, ol.OL_F32, WS, WS_BYTES,
                  stream=0)
    assert s == ol.OL_ERR_CAPACITY


# ------------------------------------------------------------------ bind


def test_bind_rejects_a_second_owner():
    ol.ol_cache_bind(CACHE, CACHE_BYTES, 11)
    try:
        ol.ol_cache_bind(CACHE, CACHE_BYTES, 11)                                  # same owner: fine
        assert status_of(ol.ol_cache_bind, CACHE + 4096, 16, 12) == ol.OL_ERR_BUSY
        desc_other = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16, owner=12)
        assert status_of(step, desc=desc_other) == ol.OL_ERR_BUSY
        desc_mine = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16, owner=11)
        assert status_of(step, desc=desc_mine) == ol.OL_ERR_INJECTED
        assert status_of(ol.ol_cache_unbind, CACHE, 12) == ol.OL_ERR_BUSY
    finally:
        ol.ol_cache_unbind(CACHE, 11)
    desc_other = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16, owner=12)
    assert status_of(step, desc=desc_other) == ol.OL_ERR_INJECTED
    ol.ol_cache_unbind(CACHE, 11)                                                # unbinding twice is fine


# ----------------------------------------------------------------- paged

P, S, M = 64, 16, 8
POOL = BASE + 128 * MB
BT = BASE + 200 * MB


def paged_desc(table, access=ol.OL_READ_WRITE):
    return ol.paged_kv(POOL, BT, np.asarray(table, np.int32), dims=(P, HKV, S, D), dtype=ol.OL_BF16, access=access)


def paged_step(table, lens):
    step(desc=paged_desc(table), updated=POOL, lens=lens, layout=ol.OL_LAYOUT_PAGED)


def test_paged_valid_and_page_checks():
    table = np.arange(B * M, dtype=np.int32).reshape(B, M)
    assert status_of(paged_step, table, (10, 128)) == ol.OL_ERR_INJECTED
    bad = table.copy()
    bad[1, 3] = P                                  # outside the pool, and reached by row 1
    assert status_of(paged_step, bad, (10, 128)) == ol.OL_ERR_PAGE
    assert status_of(paged_step, bad, (10, 48)) == ol.OL_ERR_INJECTED   # page 3 of row 1 not reached
    shared = table.copy()
    shared[1, 0] = shared[0, 0]                    # row 0 appends into page 0, which row 1 also reads
    assert status_of(paged_step, shared, (10, 20)) == ol.OL_ERR_PAGE
    assert status_of(paged_step, table, (10, 129)) == ol.OL_ERR_CAPACITY
    assert status_of(step, desc=paged_desc(table), updated=POOL + 16, lens=(1, 1),
                     layout=ol.OL_LAYOUT_PAGED) == ol.OL_ERR_ALIAS


def test_paged_cache_update_checks_slots():
    table = np.arange(B * M, dtype=np.int32).reshape(B, M)
    desc = paged_desc(table)
    assert status_of(ol.ol_paged_cache_update, desc, POOL, NEWKV, 3, [0, 125], LENS_DEV, stream=0) == \
        ol.OL_ERR_INJECTED
    assert status_of(ol.ol_paged_cache_update, desc, POOL, NEWKV, 4, [0, 125], LENS_DEV, stream=0) == \
        ol.OL_ERR_CAPACITY


# ------------------------------------------------------------------ INT4

CODES = BASE + 300 * MB
SCALES = BASE + 400 * MB
ZPS = BASE + 500 * MB


def int4_desc(d=D, **kw):
    return ol.int4_kv(CODES, SCALES, ZPS, dims=(B, HKV, C, d), **kw)


def test_int4_descriptor_rules():
    assert status_of(step, desc=int4_desc(), updated=CODES, layout=ol.OL_LAYOUT_INT4) == ol.OL_ERR_INJECTED
    assert status_of(step, desc=int4_desc(d=96), updated=CODES, layout=ol.OL_LAYOUT_INT4) == ol.OL_ERR_SHAPE
    assert status_of(step, desc=int4_desc(quant_mode=ol.OL_Q_FIXED, fixed_zp=16), updated=CODES,
                     layout=ol.OL_LAYOUT_INT4) == ol.OL_ERR_SHAPE
    assert status_of(step, desc=int4_desc(), updated=SCALES, layout=ol.OL_LAYOUT_INT4) == ol.OL_ERR_ALIAS
    overlapping = ol.int4_kv(CODES, CODES + 1024, ZPS, dims=(B, HKV, C, D))
    assert status_of(step, desc=overlapping, updated=CODES, layout=ol.OL_LAYOUT_INT4) == ol.OL_ERR_ALIAS


def test_unknown_layout():
    assert status_of(step, layout=9) == ol.OL_ERR_UNSUPPORTED


def test_history_stable_bit_keeps_write_access():
    desc = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16, access=ol.OL_READ_WRITE | ol.OL_HISTORY_STABLE)
    assert status_of(step, desc=desc) == ol.OL_ERR_INJECTED
    desc = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16, access=ol.OL_READ_ONLY | ol.OL_HISTORY_STABLE)
    assert status_of(step, desc=desc) == ol.OL_ERR_READONLY


# ------------------------------------------------- host-buffer decode step

def test_host_step_workspace_holds_the_staging():
    plain = ol.ol_workspace_size(B, HQ, HKV, D)
    host = ol.ol_workspace_size_host(B, HQ, HKV, D)
    assert host >= plain + (B * HQ * D * 4) * 2 + 2 * B * HKV * D * 4 + B * 4
    assert ol.ol_workspace_size_host(1, 7, 4, 128) == 0


def host_step(updated=CACHE, q=None, kv=None, lens=(10, 64), out=None, ws=WS, ws_bytes=None, desc=None):
    desc = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16) if desc is None else desc
    q = np.zeros((B, HQ, D), np.uint16) if q is None else q
    kv = np.zeros((2, B, HKV, 1, D), np.uint16) if kv is None else kv
    out = np.zeros((B, HQ, D), np.uint16) if out is None else out
    ws_bytes = ol.ol_workspace_size_host(B, HQ, HKV, D) if ws_bytes is None else ws_bytes
    ol.ol_decode_step_host(ol.OL_LAYOUT_CONTIGUOUS, desc, updated, q, HQ, kv, np.array(lens, np.int32), 0.0, -1,
                           out, ol.OL_BF16, ws, ws_bytes, stream=0)


def test_host_step_rejects_before_any_copy():
    # every one of these fails on the host before a copy is enqueued (no GPU here)
    assert status_of(host_step, updated=CACHE + 256) == ol.OL_ERR_ALIAS
    assert status_of(host_step, ws_bytes=ol.ol_workspace_size(B, HQ, HKV, D)) == ol.OL_ERR_WORKSPACE
    assert status_of(host_step, lens=(10, C + 1)) == ol.OL_ERR_CAPACITY
    assert status_of(host_step, lens=(0, 5)) == ol.OL_ERR_CAPACITY
    assert status_of(host_step, ws=CACHE + 64) == ol.OL_ERR_ALIAS          # staging inside the cache
    assert status_of(host_step, ws=WS + 8) == ol.OL_ERR_ALIGN
    ro = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16, access=ol.OL_READ_ONLY)
    assert status_of(host_step, desc=ro) == ol.OL_ERR_READONLY
    # y overlapping q or the new K/V in host memory
    shared = np.zeros((2, B, HQ, D), np.uint16)
    assert status_of(host_step, q=shared[0], out=shared[0]) == ol.OL_ERR_ALIAS
    assert status_of(host_step, kv=shared.reshape(-1)[: 2 * B * HKV * D].reshape(2, B, HKV, 1, D),
                     out=shared[0]) == ol.OL_ERR_ALIAS
    lib = ol.load()
    d = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16)
    import ctypes
    assert lib.ol_decode_step_host(ol.OL_LAYOUT_CONTIGUOUS, ctypes.byref(d), CACHE, None, HQ, None, None, 0.0, -1,
                                   None, ol.OL_BF16, WS, ol.ol_workspace_size_host(B, HQ, HKV, D), None) \
        == ol.OL_ERR_NULL


# ------------------------------------------------------------ chunked step

def chunk(lens=(10, 64), new_len=4, ws_bytes=None, layout=ol.OL_LAYOUT_CONTIGUOUS, desc=None, updated=CACHE):
    desc = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16) if desc is None else desc
    n = ol.ol_workspace_size_chunk(B, HQ, HKV, D, new_len) if ws_bytes is None else ws_bytes
    ol.ol_chunk_step(layout, desc, updated, Q, HQ, new_len, NEWKV, np.array(lens, np.int32), LENS_DEV, 0.0, -1, OUT,
                     ol.OL_BF16, WS, n, stream=0)


def test_chunk_step_validation():
    assert status_of(chunk) == ol.OL_ERR_INJECTED
    assert status_of(chunk, lens=(3, 64)) == ol.OL_ERR_CAPACITY          # a row shorter than the chunk
    assert status_of(chunk, lens=(10, C + 1)) == ol.OL_ERR_CAPACITY
    assert status_of(chunk, new_len=0) == ol.OL_ERR_SHAPE
    assert status_of(chunk, ws_bytes=ol.ol_workspace_size(B, HQ, HKV, D)) == ol.OL_ERR_WORKSPACE
    assert status_of(chunk, updated=CACHE + 256) == ol.OL_ERR_ALIAS
    assert status_of(chunk, desc=int4_desc(), updated=CODES, layout=ol.OL_LAYOUT_INT4) == ol.OL_ERR_INJECTED
    assert status_of(chunk, desc=int4_desc(), updated=SCALES, layout=ol.OL_LAYOUT_INT4) == ol.OL_ERR_ALIAS
    assert ol.ol_workspace_size_chunk(B, HQ, HKV, D, 4) > ol.ol_workspace_size(B, HQ, HKV, D)
