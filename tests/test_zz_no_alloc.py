"""ol_decode_step_noalloc, the decode step for callers that cannot allocate
device memory: a plugin running inside a host engine that owns all device
memory and forbids allocation while it executes, or a latency-critical decode
loop that cannot take an allocation's implicit synchronization. Its workspace
is the library's own static device scratch.

It must give, on consecutive calls that reuse that scratch, the cache bytes and
outputs the oracle gives (and what ol_decode_step gives with a caller
workspace), in every layout it takes; allocate no device memory; return
ol_decode_step's status for a rejected request with nothing enqueued; and
report a device-side guard through ol_noalloc_status.

This file is collected last so that a failure here leaves every other test run.
"""
import numpy as np
import pytest
import torch

import oracle as O
import place_kv_cache_gb300 as ol
from workloads import Workload, bf16_from_f32, block_table, contiguous_cache, make_case, poisoned_pool
from tests.gpu_util import check_out, out_as_f64, out_tensor, to_dev, to_host, workspace

pytestmark = pytest.mark.gpu


def _draw(rng, shape):
    return bf16_from_f32(rng.standard_normal(shape).astype(np.float32))


def test_noalloc_contiguous_matches_oracle_on_two_calls():
    w = Workload("noalloc", "bf16", 2, 28, 4, 128, 1024, "contiguous", seed=77)
    case = make_case(w, lens=np.array([700, 129], np.int32))
    cache = contiguous_cache(case)
    cache_ws, cache_na = to_dev(cache), to_dev(cache)
    desc_ws, desc_na = ol.kv_cache(cache_ws), ol.kv_cache(cache_na)
    ws, n = workspace(w.batch, w.q_heads, w.kv_heads, w.head_dim)
    rng = np.random.default_rng(78)
    lens = case.lens.copy()
    for call in range(2):
        q = _draw(rng, (2, 28, 128))
        kv = _draw(rng, (2, 2, 4, 1, 128))
        lens_d = to_dev(lens)
        out_ws = out_tensor(2, 28, 128, ol.OL_F32)
        out_na = out_tensor(2, 28, 128, ol.OL_F32)
        ol.ol_decode_step(ol.OL_LAYOUT_CONTIGUOUS, desc_ws, cache_ws, to_dev(q), 28, to_dev(kv), lens, lens_d, 0.0,
                          -1, out_ws, ol.OL_F32, ws, n)
        ol.ol_decode_step_noalloc(ol.OL_LAYOUT_CONTIGUOUS, desc_na, cache_na, to_dev(q), 28, to_dev(kv), lens,
                                  lens_d, 0.0, -1, out_na, ol.OL_F32)
        torch.cuda.synchronize()
        assert ol.ol_noalloc_status() == ol.OL_DEVICE_OK
        O.cache_update(cache, kv, lens - 1)
        np.testing.assert_array_equal(to_host(cache_na), cache)
        np.testing.assert_array_equal(to_host(cache_ws), cache)
        want = O.decode_attention(q, cache, lens)
        check_out(out_as_f64(out_na), want, ol.OL_F32)
        check_out(out_as_f64(out_ws), want, ol.OL_F32)
        lens = lens + 1


def test_noalloc_paged_and_int4_match_oracle_and_workspace_step():
    rng = np.random.default_rng(79)
    # paged pool, pages of 16 slots
    w = Workload("na_paged", "bf16", 3, 32, 8, 128, 16 * 16, "paged", seed=80, page_size=16, num_pages=64)
    case = make_case(w, lens=np.array([1, 100, 256], np.int32))
    table = block_table(case)
    pool = poisoned_pool(w)
    for b, h in enumerate(case.history):
        if h.shape[2]:
            O.paged_update(pool, table[b:b + 1], h[:, None], [0])
    pools = [to_dev(pool), to_dev(pool)]
    bt_d = to_dev(table)
    descs = [ol.paged_kv(p, bt_d, table) for p in pools]
    ws, n = workspace(w.batch, w.q_heads, w.kv_heads, w.head_dim)
    outs = [out_tensor(3, 32, 128, ol.OL_F32) for _ in range(2)]
    q_d, kv_d, lens_d = to_dev(case.q), to_dev(case.new_kv), to_dev(case.lens)
    ol.ol_decode_step(ol.OL_LAYOUT_PAGED, descs[0], pools[0], q_d, 32, kv_d, case.lens, lens_d, 0.0, -1, outs[0],
                      ol.OL_F32, ws, n)
    ol.ol_decode_step_noalloc(ol.OL_LAYOUT_PAGED, descs[1], pools[1], q_d, 32, kv_d, case.lens, lens_d, 0.0, -1,
                              outs[1], ol.OL_F32)
    torch.cuda.synchronize()
    assert ol.ol_noalloc_status() == ol.OL_DEVICE_OK
    O.paged_update(pool, table, case.new_kv, case.lens - 1)
    want = O.paged_attention(case.q, pool, table, case.lens)
    for p, o in zip(pools, outs):
        np.testing.assert_array_equal(to_host(p), pool)
        check_out(out_as_f64(o), want, ol.OL_F32)
    # INT4 planes, history quantized by the oracle
    w4 = Workload("na_int4", "bf16", 2, 16, 4, 128, 200, "int4", seed=81)
    case4 = make_case(w4, lens=np.array([200, 33], np.int32))
    planes = O.int4_planes(2, 4, 200, 128)
    for b, h in enumerate(case4.history):
        sub = O.int4_planes(1, 4, 200, 128)
        O.int4_append(*sub, h[:, None], [0])
        for full, part in zip(planes, sub):
            full[:, b] = part[:, 0]
    devs = [tuple(to_dev(p) for p in planes) for _ in range(2)]
    descs = [ol.int4_kv(*d, head_dim=128) for d in devs]
    ws4, n4 = workspace(2, 16, 4, 128)
    outs = [out_tensor(2, 16, 128, ol.OL_F32) for _ in range(2)]
    q_d, kv_d, lens_d = to_dev(case4.q), to_dev(case4.new_kv), to_dev(case4.lens)
    ol.ol_decode_step(ol.OL_LAYOUT_INT4, descs[0], devs[0][0], q_d, 16, kv_d, case4.lens, lens_d, 0.0, -1, outs[0],
                      ol.OL_F32, ws4, n4)
    ol.ol_decode_step_noalloc(ol.OL_LAYOUT_INT4, descs[1], devs[1][0], q_d, 16, kv_d, case4.lens, lens_d, 0.0, -1,
                              outs[1], ol.OL_F32)
    torch.cuda.synchronize()
    assert ol.ol_noalloc_status() == ol.OL_DEVICE_OK
    O.int4_append(*planes, case4.new_kv, case4.lens - 1)
    want = O.int4_attention(case4.q, *planes, case4.lens, cur_kv=case4.new_kv)
    for d, o in zip(devs, outs):
        for g, r in zip(d, planes):
            np.testing.assert_array_equal(to_host(g), r)
        check_out(out_as_f64(o), want, ol.OL_F32)


def test_noalloc_allocates_no_device_memory():
    w = Workload("na_mem", "bf16", 4, 32, 8, 128, 512, "contiguous", seed=82)
    case = make_case(w, lens=np.array([512, 300, 17, 1], np.int32))
    cache_d = to_dev(contiguous_cache(case))
    desc = ol.kv_cache(cache_d)
    q_d, kv_d, lens_d = to_dev(case.q), to_dev(case.new_kv), to_dev(case.lens)
    out = out_tensor(4, 32, 128, ol.OL_BF16)
    step = lambda: ol.ol_decode_step_noalloc(ol.OL_LAYOUT_CONTIGUOUS, desc, cache_d, q_d, 32, kv_d, case.lens, lens_d,
                                             0.0, -1, out, ol.OL_BF16)
    step()                                   # warm-up: module and scratch address set up on this device
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    for _ in range(16):
        step()
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_rejects_as_the_workspace_step_does():
    # the scratch size: a batch whose worst-case workspace exceeds it, rejected before any launch
    batch, q_heads, kv_heads, head_dim = 4096, 8, 8, 128
    assert ol.ol_workspace_size(batch, q_heads, kv_heads, head_dim) > 16 * 1024 * 1024
    cache = torch.zeros(16, dtype=torch.bfloat16, device="cuda:0")
    big = ol.kv_cache(cache, dims=(batch, kv_heads, 16, head_dim), dtype=ol.OL_BF16)
    q = torch.zeros(16, dtype=torch.bfloat16, device="cuda:0")
    before = cache.clone()
    with pytest.raises(ol.OlError) as e:
        ol.ol_decode_step_noalloc(ol.OL_LAYOUT_CONTIGUOUS, big, cache, q, q_heads, q, np.ones(batch, np.int32), q,
                                  0.0, -1, q, ol.OL_F32)
    assert e.value.status == ol.OL_ERR_WORKSPACE
    # other rejections: the status ol_decode_step returns for the same request, the cache untouched
    w = Workload("na_rej", "bf16", 2, 8, 2, 128, 64, "contiguous", seed=83)
    case = make_case(w, lens=np.array([10, 64], np.int32))
    cache_d = to_dev(contiguous_cache(case))
    snap = cache_d.clone()
    desc = ol.kv_cache(cache_d)
    ro = ol.kv_cache(cache_d, access=ol.OL_READ_ONLY)
    other = torch.empty_like(cache_d)
    q_d, kv_d = to_dev(case.q), to_dev(case.new_kv)
    ws, n = workspace(2, 8, 2, 128)
    out = out_tensor(2, 8, 128, ol.OL_F32)
    over = np.array([10, 65], np.int32)
    bad = [(desc, other, case.lens, "alias"), (ro, cache_d, case.lens, "read-only"), (desc, cache_d, over, "capacity")]
    for d, upd, lens, what in bad:
        with pytest.raises(ol.OlError) as e1:
            ol.ol_decode_step(ol.OL_LAYOUT_CONTIGUOUS, d, upd, q_d, 8, kv_d, lens, to_dev(lens), 0.0, -1, out,
                              ol.OL_F32, ws, n)
        with pytest.raises(ol.OlError) as e2:
            ol.ol_decode_step_noalloc(ol.OL_LAYOUT_CONTIGUOUS, d, upd, q_d, 8, kv_d, lens, to_dev(lens), 0.0, -1, out,
                                      ol.OL_F32)
        assert e1.value.status == e2.value.status, what
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(cache_d), to_host(snap))    # bit patterns (the spare rows hold NaN)
    assert torch.equal(cache, before)


def test_noalloc_status_reports_a_device_guard():
    # 200 rows: the lengths are read from device memory; row 5's device length
    # exceeds the capacity, so the kernels clamp it and record OL_DEVICE_GUARD
    B, Hq, Hkv, D, C = 200, 8, 2, 128, 64
    w = Workload("na_guard", "bf16", B, Hq, Hkv, D, C, "contiguous", seed=84)
    lens = np.full(B, 33, np.int32)
    case = make_case(w, lens=lens)
    cache_d = to_dev(contiguous_cache(case))
    desc = ol.kv_cache(cache_d)
    q_d, kv_d = to_dev(case.q), to_dev(case.new_kv)
    out = out_tensor(B, Hq, D, ol.OL_F32)
    lens_bad = lens.copy()
    lens_bad[5] = C + 7
    ol.ol_decode_step_noalloc(ol.OL_LAYOUT_CONTIGUOUS, desc, cache_d, q_d, Hq, kv_d, lens, to_dev(lens_bad), 0.0, -1,
                              out, ol.OL_F32)
    assert ol.ol_noalloc_status() == ol.OL_DEVICE_GUARD
    assert ol.ol_noalloc_status() == ol.OL_DEVICE_OK                  # read and cleared
    # the next call starts from cleared counters: a consistent call is correct again
    cache2 = contiguous_cache(case)
    cache2_d = to_dev(cache2)
    ol.ol_decode_step_noalloc(ol.OL_LAYOUT_CONTIGUOUS, ol.kv_cache(cache2_d), cache2_d, q_d, Hq, kv_d, lens,
                              to_dev(lens), 0.0, -1, out, ol.OL_F32)
    assert ol.ol_noalloc_status() == ol.OL_DEVICE_OK
    O.cache_update(cache2, case.new_kv, lens - 1)
    np.testing.assert_array_equal(to_host(cache2_d), cache2)
    check_out(out_as_f64(out), O.decode_attention(case.q, cache2, lens), ol.OL_F32)
