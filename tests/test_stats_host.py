"""CPU tests of the per-call storage statistics (ol_stats). Calls stop right
after validation (host fault injection), which is where the library records
them, so no GPU is needed. Expected counts are written from the definitions
of the counters (page "Persistent input/output feedback", sections Opt-in
storage auditing through runtime events and Optional heterogeneous paged KV),
and one is the pages' own figure for a FLOAT append."""
import numpy as np
import pytest

import place_kv_cache_gb300 as ol
from tests.test_abi_host import (B, BASE, C, CACHE, CODES, D, HKV, HQ, LENS_DEV, MB, NEWKV, OUT, Q, WS, WS_BYTES,
                                 int4_desc, status_of, step)


@pytest.fixture(autouse=True)
def _inject(monkeypatch):
    monkeypatch.setenv("OL_FAULT_INJECT", "after_validate")
    ol.ol_reset_stats()
    yield


def test_float_append_copies_four_bytes_per_element_and_no_prefix():
    # "For one new token with FLOAT K/V head sizes Dk and Dv, appending copies
    # 4 * (Dk + Dv) bytes"; reuse within capacity allocates nothing and copies
    # no prefix bytes. Here B = 1, one kv head, Dk = Dv = 4 (an fp32 cache).
    desc = ol.kv_cache(CACHE, dims=(1, 1, 16, 4), dtype=ol.OL_F32)
    assert status_of(ol.ol_cache_update, desc, CACHE, NEWKV, 1, 7, stream=0) == ol.OL_ERR_INJECTED
    s = ol.ol_last_call_stats()
    assert s["storage_append_copied_bytes"] == 4 * (4 + 4)
    assert s["storage_prefix_copied_bytes"] == 0
    assert s["storage_allocations"] == 0 and s["storage_allocated_bytes"] == 0
    assert s["storage_reuse_count"] == 2 and s["calls"] == 1


def test_decode_step_counts():
    lens = (10, 64)
    assert status_of(step, lens=lens) == ol.OL_ERR_INJECTED
    s = ol.ol_last_call_stats()
    hist = (10 - 1) + (64 - 1)                     # the current token comes from new_kv
    assert s["attended_tokens"] == (10 + 64) * HKV
    assert s["kv_payload_bytes_read"] == 2 * hist * HKV * D * 2
    assert s["storage_append_copied_bytes"] == 2 * B * HKV * D * 2
    assert s["dequantized_bytes"] == 0
    assert s["storage_prefix_copied_bytes"] == 0 and s["storage_allocations"] == 0
    assert s["workspace_bytes"] == WS_BYTES


def test_window_limits_the_visible_tokens():
    def windowed():
        desc = ol.kv_cache(CACHE, dims=(B, HKV, C, D), dtype=ol.OL_BF16)
        ol.ol_decode_attention(desc, Q, HQ, np.array([10, 64], np.int32), LENS_DEV, 0.0, 5, OUT, ol.OL_BF16, WS,
                               WS_BYTES, stream=0)
    assert status_of(windowed) == ol.OL_ERR_INJECTED
    s = ol.ol_last_call_stats()
    assert s["attended_tokens"] == (6 + 6) * HKV           # the last token and the 5 before it
    assert s["kv_payload_bytes_read"] == 2 * 12 * HKV * D * 2  # no new_kv: every visible token from the cache
    assert s["storage_append_copied_bytes"] == 0 and s["storage_reuse_count"] == 0


def test_int4_step_counts_dequantized_float_bytes():
    assert status_of(step, desc=int4_desc(), updated=CODES, layout=ol.OL_LAYOUT_INT4, lens=(3, 40)) == \
        ol.OL_ERR_INJECTED
    s = ol.ol_last_call_stats()
    hist = 2 + 39
    per_token = D // 2 + (D // 32) * 2 + D // 64         # codes + fp16 scales + zero-point nibbles
    assert s["kv_payload_bytes_read"] == 2 * hist * HKV * per_token
    assert s["dequantized_bytes"] == 2 * hist * HKV * D * 4
    assert s["storage_append_copied_bytes"] == 2 * B * HKV * per_token


def test_totals_accumulate_and_failed_validation_records_nothing():
    assert status_of(step, lens=(10, 64)) == ol.OL_ERR_INJECTED
    first = ol.ol_last_call_stats()
    assert status_of(step, lens=(5, 5)) == ol.OL_ERR_INJECTED
    assert status_of(step, lens=(5, C + 1)) == ol.OL_ERR_CAPACITY   # rejected: not recorded
    last = ol.ol_last_call_stats()
    assert last["attended_tokens"] == 10 * HKV
    tot = ol.ol_total_stats()
    assert tot["calls"] == 2
    assert tot["attended_tokens"] == first["attended_tokens"] + last["attended_tokens"]
    ol.ol_reset_stats()
    assert ol.ol_total_stats()["calls"] == 0 and ol.ol_last_call_stats()["calls"] == 0
