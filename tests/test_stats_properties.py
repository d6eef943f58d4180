"""Randomised CPU tests of the per-call storage statistics (ol_stats) of the
decode step and of attention alone, over drawn shapes, dtypes, lengths and
windows. Expected counts are written from the counters' definitions: the
visible range of the query at p = lens - 1 is [max(0, p - w), p] (or [0, p]);
a fused step takes the current token from new_kv, so it reads one token
fewer from the cache than it attends, and stores one token per (row, kv
head, plane); nothing is ever allocated or copied from the prefix. Calls stop
right after validation (host fault injection), where the library records
them: no GPU is needed.
"""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import place_kv_cache_gb300 as ol  # noqa: E402

BASE = 0x7D0000000000
GB = 1 << 30


@pytest.fixture(autouse=True)
def _inject(monkeypatch):
    monkeypatch.setenv("OL_FAULT_INJECT", "after_validate")
    yield


@st.composite
def calls(draw):
    B = draw(st.integers(1, 5))
    Hkv = draw(st.integers(1, 4))
    G = draw(st.integers(1, 4))
    D = draw(st.sampled_from([64, 128]))
    dtype = draw(st.sampled_from([ol.OL_BF16, ol.OL_F32]))
    C = draw(st.integers(1, 5000))
    lens = draw(st.lists(st.integers(1, C), min_size=B, max_size=B))
    window = draw(st.sampled_from([-1, 0, 1, 7, 100, 4096]))
    fused = draw(st.booleans())
    return B, Hkv, G, D, dtype, C, np.array(lens, np.int32), window, fused


def visible(n, window):
    p = n - 1
    return n if window < 0 else p - max(0, p - window) + 1


@settings(max_examples=200, deadline=None, derandomize=True)
@given(calls())
def test_counts_follow_their_definitions(c):
    B, Hkv, G, D, dtype, C, lens, window, fused = c
    elt = 2 if dtype == ol.OL_BF16 else 4
    cache = BASE
    q, new_kv, out, lens_dev, ws = (BASE + k * GB for k in (1, 2, 3, 4, 5))
    ws_bytes = ol.ol_workspace_size(B, Hkv * G, Hkv, D)
    desc = ol.kv_cache(cache, dims=(B, Hkv, C, D), dtype=dtype)
    ol.ol_reset_stats()
    with pytest.raises(ol.OlError) as e:
        if fused:
            ol.ol_decode_step(ol.OL_LAYOUT_CONTIGUOUS, desc, cache, q, Hkv * G, new_kv, lens, lens_dev, 0.0, window,
                              out, ol.OL_BF16, ws, ws_bytes, stream=0)
        else:
            ol.ol_decode_attention(desc, q, Hkv * G, lens, lens_dev, 0.0, window, out, ol.OL_BF16, ws, ws_bytes,
                                   stream=0)
    assert e.value.status == ol.OL_ERR_INJECTED
    s = ol.ol_last_call_stats()
    vis = [visible(int(n), window) for n in lens]
    from_cache = sum(v - (1 if fused else 0) for v in vis)
    assert s["calls"] == 1
    assert s["attended_tokens"] == sum(vis) * Hkv
    assert s["kv_payload_bytes_read"] == 2 * from_cache * Hkv * D * elt
    assert s["storage_append_copied_bytes"] == (2 * B * Hkv * D * elt if fused else 0)
    assert s["storage_reuse_count"] == (2 if fused else 0)
    assert s["storage_prefix_copied_bytes"] == 0
    assert s["storage_allocations"] == 0 and s["storage_allocated_bytes"] == 0
    assert s["dequantized_bytes"] == 0
    assert s["workspace_bytes"] <= ws_bytes
    tot = ol.ol_total_stats()
    assert tot["calls"] == 1 and tot["attended_tokens"] == s["attended_tokens"]
