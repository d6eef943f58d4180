"""CPU tests of the heterogeneous paged cache's C ABI: descriptor layout,
host validation of formats, pages and aliasing, and the host format mirror.

No GPU is touched: device pointers are fake aligned addresses that host
validation compares but never dereferences, and valid requests stop right
after validation through the host fault-injection switch (OL_FAULT_INJECT).
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

import place_kv_cache_gb300 as ol

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE = 0x7F0000000000
MB = 1 << 20
B, HQ, HKV, S, M, D = 2, 8, 2, 16, 8, 128
P = B * M
SLOT = 2 * HKV * S * D * 4
POOL = BASE
FMT_DEV = BASE + 200 * MB
BT_DEV = BASE + 201 * MB
Q = BASE + 210 * MB
NEWKV = BASE + 211 * MB
OUT = BASE + 212 * MB
LENS_DEV = BASE + 213 * MB
WS = BASE + 214 * MB
WS_BYTES = ol.ol_workspace_size(B, HQ, HKV, D)

BF16 = (ol.OL_FMT_BF16, 1.0, 0)
I8 = (ol.OL_FMT_I8, 0.03125, 0)
U4 = (ol.OL_FMT_U4, 0.5, 8)


@pytest.fixture(autouse=True)
def _inject(monkeypatch):
    monkeypatch.setenv("OL_FAULT_INJECT", "after_validate")
    yield


def status_of(fn, *a, **k):
    try:
        fn(*a, **k)
    except ol.OlError as e:
        return e.status
    return ol.OL_OK


def mirror(fmt=(BF16, BF16)):
    m = np.zeros(P, ol.PAGE_FORMAT_DTYPE)
    m["kf"], m["ks"], m["kz"] = fmt[0]
    m["vf"], m["vs"], m["vz"] = fmt[1]
    return m


def desc(m=None, table=None, access=ol.OL_READ_WRITE, head_dim=D, pool=POOL, fmt_dev=FMT_DEV, page_size=S):
    m = mirror() if m is None else m
    table = np.arange(P, dtype=np.int32).reshape(B, M) if table is None else table
    return ol.hpaged_kv(pool, fmt_dev, m, BT_DEV, table, kv_heads=HKV, page_size=page_size, head_dim=head_dim,
                        access=access)


def step(d=None, lens=(10, 100), new_pages=None, updated=POOL, q=Q, window=-1):
    d = desc() if d is None else d
    ol.ol_hpaged_decode_step(d, updated, q, HQ, NEWKV, ol.page_format() if new_pages is None else new_pages,
                             np.array(lens, np.int32), LENS_DEV, 0.0, window, OUT, ol.OL_BF16, WS, WS_BYTES, stream=0)


def attend(d=None, lens=(10, 100), cur=None, window=-1):
    d = desc() if d is None else d
    ol.ol_hpaged_decode_attention(d, Q, HQ, np.array(lens, np.int32), LENS_DEV, cur, 0.0, window, OUT, ol.OL_F32, WS,
                                  WS_BYTES, stream=0)


def append(d=None, pos=(0, 16), new_len=4, new_pages=None, updated=POOL):
    d = desc() if d is None else d
    ol.ol_hpaged_append(d, updated, NEWKV, new_len, np.array(pos, np.int32), LENS_DEV,
                        ol.page_format() if new_pages is None else new_pages, stream=0)


def quantize(d=None, pages=(1, 5), valid=(16, 3), to=None, updated=POOL):
    d = desc() if d is None else d
    ol.ol_hpaged_quantize(d, updated, np.array(pages, np.int32), LENS_DEV, np.array(valid, np.int32), LENS_DEV + 4096,
                          ol.page_format(k=I8, v=U4) if to is None else to, stream=0)


def test_struct_layout_matches_the_header():
    src = r'''
#include <stddef.h>
#include <stdio.h>
#include "ol.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu\n", sizeof(ol_hpaged_kv), sizeof(ol_page_format), sizeof(ol_plane_format),
         offsetof(ol_hpaged_kv, num_pages), offsetof(ol_hpaged_kv, owner), offsetof(ol_page_format, v),
         offsetof(ol_plane_format, zero_point));
  return 0;
}
'''
    with tempfile.TemporaryDirectory() as t:
        c, exe = os.path.join(t, "l.c"), os.path.join(t, "l")
        with open(c, "w") as f:
            f.write(src)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        got = [int(x) for x in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    want = [ctypes.sizeof(ol.HPagedKV), ctypes.sizeof(ol.PageFormat), ctypes.sizeof(ol.PlaneFormat),
            ol.HPagedKV.num_pages.offset, ol.HPagedKV.owner.offset, ol.PageFormat.v.offset,
            ol.PlaneFormat.zero_point.offset]
    assert got == want
    assert ol.PAGE_FORMAT_DTYPE.itemsize == ctypes.sizeof(ol.PageFormat)


def test_valid_calls_pass_validation():
    assert status_of(step) == ol.OL_ERR_INJECTED
    assert status_of(attend) == ol.OL_ERR_INJECTED
    assert status_of(attend, cur=NEWKV) == ol.OL_ERR_INJECTED
    assert status_of(append) == ol.OL_ERR_INJECTED
    assert status_of(quantize) == ol.OL_ERR_INJECTED


def test_generic_entry_points_do_not_take_the_layout():
    d = desc()
    assert status_of(ol.ol_decode_step, ol.OL_LAYOUT_HPAGED, d, POOL, Q, HQ, NEWKV, np.array([3, 3], np.int32),
                     LENS_DEV, 0.0, -1, OUT, ol.OL_BF16, WS, WS_BYTES, stream=0) == ol.OL_ERR_UNSUPPORTED
    assert status_of(ol.ol_chunk_step, ol.OL_LAYOUT_HPAGED, d, POOL, Q, HQ, 2, NEWKV, np.array([3, 3], np.int32),
                     LENS_DEV, 0.0, -1, OUT, ol.OL_BF16, WS, WS_BYTES, stream=0) == ol.OL_ERR_UNSUPPORTED


def test_descriptor_rules():
    assert status_of(step, d=desc(head_dim=126)) == ol.OL_ERR_SHAPE            # head_dim % 4
    assert status_of(step, d=desc(pool=POOL + 8), updated=POOL + 8) == ol.OL_ERR_ALIGN
    assert status_of(step, d=desc(fmt_dev=POOL + SLOT)) == ol.OL_ERR_ALIAS        # table inside the pool
    assert status_of(step, updated=POOL + 16) == ol.OL_ERR_ALIAS
    assert status_of(step, d=desc(access=ol.OL_READ_ONLY)) == ol.OL_ERR_READONLY
    assert status_of(attend, d=desc(access=ol.OL_READ_ONLY)) == ol.OL_ERR_INJECTED
    assert status_of(step, q=FMT_DEV) == ol.OL_ERR_ALIAS                          # q over the format table
    with pytest.raises(TypeError):
        ol.hpaged_kv(POOL, FMT_DEV, np.zeros(P, np.int32), BT_DEV, np.zeros((B, M), np.int32), kv_heads=HKV,
                     page_size=S, head_dim=D)


@pytest.mark.parametrize("bad", [(ol.OL_FMT_I8, 0.0, 0), (ol.OL_FMT_U4, 0.5, 16), (ol.OL_FMT_I2, 1.0, -3),
                                 (9, 1.0, 0), (-1, 1.0, 0), (ol.OL_FMT_U8, float("inf"), 0),
                                 (ol.OL_FMT_I4, float("nan"), 0)])
def test_invalid_formats_are_rejected(bad):
    assert status_of(step, new_pages=ol.page_format(k=bad)) == ol.OL_ERR_SHAPE
    assert status_of(append, new_pages=ol.page_format(v=bad)) == ol.OL_ERR_SHAPE
    assert status_of(quantize, to=ol.page_format(k=bad)) == ol.OL_ERR_SHAPE
    # a page read with a bad format, and one outside the visible window
    m = mirror()
    m["kf"][3] = bad[0]
    m["ks"][3] = bad[1]
    m["kz"][3] = bad[2]
    if bad[0] in range(3):   # dense formats ignore scale and zero point
        return
    assert status_of(attend, d=desc(m), lens=(60, 5)) == ol.OL_ERR_SHAPE          # row 0 reads page 3
    assert status_of(attend, d=desc(m), lens=(40, 5)) == ol.OL_ERR_INJECTED        # pages 0..2 only
    assert status_of(attend, d=desc(m), lens=(128, 5), window=70) == ol.OL_ERR_SHAPE      # 57..127: from page 3
    assert status_of(attend, d=desc(m), lens=(128, 5), window=60) == ol.OL_ERR_INJECTED   # 67..127: from page 4


def test_append_formats_of_started_and_continued_pages():
    m = mirror()
    m["vf"][3] = 42                               # page 3 (row 0, tokens 48..63) holds no valid format
    # an append that starts page 3 gives it the new formats: accepted
    assert status_of(append, d=desc(m), pos=(48, 0), new_len=5) == ol.OL_ERR_INJECTED
    assert status_of(step, d=desc(m), lens=(49, 3)) == ol.OL_ERR_INJECTED
    # an append that continues page 3 needs its formats
    assert status_of(append, d=desc(m), pos=(50, 0), new_len=1) == ol.OL_ERR_SHAPE
    assert status_of(step, d=desc(m), lens=(51, 3)) == ol.OL_ERR_SHAPE
    # attention with the current token from cur_kv does not read page 3 at lens 49
    assert status_of(attend, d=desc(m), lens=(49, 3), cur=NEWKV) == ol.OL_ERR_INJECTED
    assert status_of(attend, d=desc(m), lens=(49, 3)) == ol.OL_ERR_SHAPE


def test_pages_capacity_and_sharing():
    table = np.arange(P, dtype=np.int32).reshape(B, M)
    assert status_of(step, lens=(128, 1)) == ol.OL_ERR_INJECTED
    assert status_of(step, lens=(129, 1)) == ol.OL_ERR_CAPACITY
    assert status_of(step, lens=(0, 1)) == ol.OL_ERR_CAPACITY
    bad = table.copy()
    bad[1, 2] = P
    assert status_of(step, d=desc(table=bad), lens=(5, 40)) == ol.OL_ERR_PAGE
    assert status_of(step, d=desc(table=bad), lens=(5, 30)) == ol.OL_ERR_INJECTED
    shared = table.copy()
    shared[1, 0] = shared[0, 0]
    assert status_of(step, d=desc(table=shared), lens=(5, 20)) == ol.OL_ERR_PAGE
    assert status_of(append, pos=(125, 0), new_len=4) == ol.OL_ERR_CAPACITY
    assert status_of(attend, lens=(0, 1), cur=NEWKV) == ol.OL_ERR_CAPACITY


def test_quantize_checks():
    assert status_of(quantize, pages=(1, 1), valid=(2, 2)) == ol.OL_ERR_SHAPE     # duplicate
    assert status_of(quantize, pages=(P, 1)) == ol.OL_ERR_PAGE
    assert status_of(quantize, pages=(-1, 1)) == ol.OL_ERR_PAGE
    assert status_of(quantize, valid=(17, 0)) == ol.OL_ERR_CAPACITY
    assert status_of(quantize, valid=(-1, 0)) == ol.OL_ERR_CAPACITY
    assert status_of(quantize, updated=POOL + 16) == ol.OL_ERR_ALIAS
    assert status_of(quantize, d=desc(access=ol.OL_READ_ONLY)) == ol.OL_ERR_READONLY
    m = mirror()
    m["kf"][5] = 11
    assert status_of(quantize, d=desc(m)) == ol.OL_ERR_SHAPE                      # page 5 cannot be decoded
    assert status_of(quantize, pages=(), valid=()) == ol.OL_ERR_INJECTED
    big = desc(page_size=512)
    assert status_of(quantize, d=big, valid=(1, 1)) == ol.OL_ERR_UNSUPPORTED        # 512 x 128 fp32 > 200 KB


def test_rejected_and_injected_calls_leave_the_mirror():
    m = mirror((I8, U4))
    before = m.copy()
    for fn, kw in ((append, {"pos": (0, 16)}), (step, {"lens": (17, 33)}), (quantize, {})):
        assert status_of(fn, d=desc(m), **kw) == ol.OL_ERR_INJECTED
        assert status_of(fn, d=desc(m), updated=POOL + 16, **kw) == ol.OL_ERR_ALIAS
    np.testing.assert_array_equal(m, before)


def test_statistics_follow_the_page_formats():
    m = mirror()
    m["kf"][:M], m["ks"][:M], m["kz"][:M] = I8      # row 0: K INT8 (128 B rows), V BFLOAT16 (256 B rows)
    m["vf"][M:], m["vs"][M:], m["vz"][M:] = U4      # row 1: K BFLOAT16, V UINT4 (64 B rows)
    ol.ol_reset_stats()
    assert status_of(step, d=desc(m), lens=(33, 18), new_pages=ol.page_format(k=I8, v=U4)) == ol.OL_ERR_INJECTED
    s = ol.ol_last_call_stats()
    hist = {0: 32, 1: 17}
    assert s["attended_tokens"] == (33 + 18) * HKV
    assert s["kv_payload_bytes_read"] == HKV * (hist[0] * (128 + 256) + hist[1] * (256 + 64))
    assert s["dequantized_bytes"] == HKV * (hist[0] + hist[1]) * D * 4
    # row 0 starts page 2 at token 32 (new formats I8 / U4); row 1 continues page 1 at 17 (BF16 / U4)
    assert s["storage_append_copied_bytes"] == HKV * ((128 + 64) + (256 + 64))
    assert s["storage_allocations"] == 0 and s["storage_prefix_copied_bytes"] == 0


def chunk(d=None, lens=(10, 100), new_len=4, new_pages=None, updated=POOL, window=-1, ws_bytes=None):
    d = desc() if d is None else d
    n = ol.ol_workspace_size_chunk(B, HQ, HKV, D, new_len) if ws_bytes is None else ws_bytes
    ol.ol_hpaged_chunk_step(d, updated, Q, HQ, new_len, NEWKV, ol.page_format() if new_pages is None else new_pages,
                            np.array(lens, np.int32), LENS_DEV, 0.0, window, OUT, ol.OL_BF16, WS, n, stream=0)


def test_chunk_step_validation():
    assert status_of(chunk) == ol.OL_ERR_INJECTED
    assert status_of(chunk, lens=(3, 100)) == ol.OL_ERR_CAPACITY          # a row shorter than the chunk
    assert status_of(chunk, lens=(10, M * S + 1)) == ol.OL_ERR_CAPACITY
    assert status_of(chunk, new_len=0) == ol.OL_ERR_SHAPE
    assert status_of(chunk, ws_bytes=WS_BYTES) == ol.OL_ERR_WORKSPACE      # the decode step's size is too small
    assert status_of(chunk, updated=POOL + 16) == ol.OL_ERR_ALIAS
    assert status_of(chunk, d=desc(access=ol.OL_READ_ONLY)) == ol.OL_ERR_READONLY
    assert status_of(chunk, new_pages=ol.page_format(k=(ol.OL_FMT_U4, 0.5, 16))) == ol.OL_ERR_SHAPE
    m = mirror()
    m["vf"][2] = 42                           # row 0's page 2 (tokens 32..47)
    assert status_of(chunk, d=desc(m), lens=(36, 5)) == ol.OL_ERR_INJECTED  # the chunk 32..35 starts page 2
    assert status_of(chunk, d=desc(m), lens=(40, 5)) == ol.OL_ERR_SHAPE     # 32..35 are history: page 2 is read
    assert status_of(chunk, d=desc(m), lens=(40, 8), new_len=8) == ol.OL_ERR_INJECTED  # 32..39 start page 2
    np.testing.assert_array_equal(m["vf"][2], 42)                          # validation never touches the mirror
