"""Parity at the full workload sizes, in the launch configuration bench.py
times (the default plan, history-stable caches), against the CPU oracle.

Every full-size step runs twice on the same inputs: with a bf16 output (the
tolerance adds half a bf16 ulp of y) and with an fp32 output, held to the
plain max-abs-error bound of 2e-3. The second run repeats the append at the
same positions with the same values, so the cache is the same after both and
is compared byte for byte. Outputs are compared on every row where the oracle
finishes in seconds (the oracle is C; its calls run on host threads, one row
each), else on rows that include the shortest, the longest and the median
length.

Inputs follow the seeded recipe of each workload (workloads.WORKLOADS); the
cache history is laid out, paged or quantized by the oracle-side helpers, never
by the CUDA path.
"""
import concurrent.futures
import os

import numpy as np
import pytest
import torch

import oracle as O
import place_kv_cache_gb300 as ol
from workloads import (AGE_FORMATS, WORKLOADS, bf16_from_f32, block_table, contiguous_cache, make_case,
                       page_format_classes, poisoned_pool)
from tests.gpu_util import check_out, out_as_f64, out_tensor, to_dev, to_host, workspace

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL = 2e-3
# the access bits bench.py gives its non-chained caches: history rows stable,
# so the first K/V tiles are requested before the dependency wait
STABLE = ol.OL_READ_WRITE | ol.OL_HISTORY_STABLE
OUTS = ((ol.OL_BF16, torch.bfloat16), (ol.OL_F32, torch.float32))


def threaded(fn, items):
    """fn over items on host threads (the oracle releases the GIL)."""
    n = max(1, min(len(items), len(os.sched_getaffinity(0)), 32))
    with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
        return list(ex.map(fn, items))


def check(got, want, out_dtype):
    """bf16 outputs: 2e-3 plus half a bf16 ulp per element; fp32: max |err| <= 2e-3."""
    if out_dtype == ol.OL_F32:
        err = float(np.max(np.abs(got - want))) if got.size else 0.0
        assert err <= TOL, f"max abs error {err:.3e} > {TOL}"
        return err
    return check_out(got, want, out_dtype)


def spread_rows(lens, extra=()):
    """Row indices with the shortest, longest and median lengths, plus `extra`."""
    order = np.argsort(lens, kind="stable")
    return sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2]), *[int(e) for e in extra]})


def _pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def _contiguous_want(case, cache):
    """Oracle outputs of every row, one row per thread."""
    w = case.workload

    def row(b):
        return O.decode_attention(case.q[b:b + 1], np.ascontiguousarray(cache[:, b:b + 1]), case.lens[b:b + 1])[0]
    return np.stack(threaded(row, list(range(w.batch))))


@pytest.mark.parametrize("host", [False, True], ids=["device_buffers", "host_buffers"])
@pytest.mark.parametrize("name", ["qwen_b1_gqa7", "ragged_b32"])
def test_contiguous_full_size(name, host):
    w = WORKLOADS[name]
    case = make_case(w)
    cache = contiguous_cache(case)
    cache_d = to_dev(cache)
    desc = ol.kv_cache(cache_d, access=STABLE)
    got = {}
    if host:  # the host-buffer call bench.py's e2e times: pinned q, new K/V and y used in place
        n = ol.ol_workspace_size_host(w.batch, w.q_heads, w.kv_heads, w.head_dim)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        ol.ol_workspace_init(ws, n)
        for code, dt in OUTS:
            out = torch.full((w.batch, w.q_heads, w.head_dim), float("nan"), dtype=dt).pin_memory()
            ol.ol_decode_step_host(ol.OL_LAYOUT_CONTIGUOUS, desc, cache_d, _pinned(case.q), w.q_heads,
                                   _pinned(case.new_kv), torch.from_numpy(case.lens), 0.0, -1, out, code, ws, n)
            torch.cuda.synchronize()
            got[code] = out_as_f64(out)
    else:
        ws, n = workspace(w.batch, w.q_heads, w.kv_heads, w.head_dim)
        q_d, kv_d, lens_d = to_dev(case.q), to_dev(case.new_kv), to_dev(case.lens)
        for code, _ in OUTS:
            out = out_tensor(w.batch, w.q_heads, w.head_dim, code)
            ol.ol_decode_step(ol.OL_LAYOUT_CONTIGUOUS, desc, cache_d, q_d, w.q_heads, kv_d, case.lens, lens_d, 0.0,
                              -1, out, code, ws, n)
            torch.cuda.synchronize()
            got[code] = out_as_f64(out)
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    O.cache_update(cache, case.new_kv, case.lens - 1)          # the expected cache, in place
    np.testing.assert_array_equal(to_host(cache_d), cache)
    del cache_d
    want = _contiguous_want(case, cache)
    for code, _ in OUTS:
        check(got[code], want, code)


def test_paged_full_size_every_row():
    w = WORKLOADS["paged_b64"]
    case = make_case(w)
    table = block_table(case)
    pool = poisoned_pool(w)

    def fill(b):  # rows own disjoint pages
        h = case.history[b]
        if h.shape[2]:
            O.paged_update(pool, table[b:b + 1], h[:, None], [0])
    threaded(fill, list(range(w.batch)))
    case.history = None                                        # free the host copy of the history
    pool_d = to_dev(pool)
    bt_d = to_dev(table)
    ws, n = workspace(w.batch, w.q_heads, w.kv_heads, w.head_dim)
    desc = ol.paged_kv(pool_d, bt_d, table, access=STABLE)
    q_d, kv_d, lens_d = to_dev(case.q), to_dev(case.new_kv), to_dev(case.lens)
    got = {}
    for code, _ in OUTS:
        out = out_tensor(w.batch, w.q_heads, w.head_dim, code)
        ol.ol_decode_step(ol.OL_LAYOUT_PAGED, desc, pool_d, q_d, w.q_heads, kv_d, case.lens, lens_d, 0.0, -1, out,
                          code, ws, n)
        torch.cuda.synchronize()
        got[code] = out_as_f64(out)
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    O.paged_update(pool, table, case.new_kv, case.lens - 1)
    np.testing.assert_array_equal(to_host(pool_d), pool)      # every pool byte
    del pool_d

    def row(b):
        return O.paged_attention(case.q[b:b + 1], pool, table[b:b + 1], case.lens[b:b + 1])[0]
    want = np.stack(threaded(row, list(range(w.batch))))
    for code, _ in OUTS:
        check(got[code], want, code)


def test_int4_full_size_chained():
    # 64 chained steps at capacity 32768, history of 16384 tokens quantized by
    # the oracle; every row compared at 8 steps spread over the chain
    w = WORKLOADS["int4_b16"]
    case = make_case(w)

    def quantized(b):
        sub = O.int4_planes(1, w.kv_heads, w.capacity, w.head_dim)
        O.int4_append(*sub, case.history[b][:, None], [0])
        return sub
    subs = threaded(quantized, list(range(w.batch)))
    planes = O.int4_planes(w.batch, w.kv_heads, w.capacity, w.head_dim)
    for b, sub in enumerate(subs):
        for full, part in zip(planes, sub):
            full[:, b] = part[:, 0]
    del subs
    case.history = None
    dplanes = tuple(to_dev(p) for p in planes)
    desc = ol.int4_kv(*dplanes, head_dim=w.head_dim)
    ws, n = workspace(w.batch, w.q_heads, w.kv_heads, w.head_dim)
    rng = np.random.default_rng(w.seed + 1)
    lens = case.lens.copy()
    compared = (0, 9, 18, 27, 36, 45, 54, w.steps - 1)
    for step in range(w.steps):
        q = bf16_from_f32(rng.standard_normal((w.batch, w.q_heads, w.head_dim)).astype(np.float32))
        kv = bf16_from_f32(rng.standard_normal((2, w.batch, w.kv_heads, 1, w.head_dim)).astype(np.float32))
        q_d, kv_d, lens_d = to_dev(q), to_dev(kv), to_dev(lens)
        got = {}
        for code, _ in (OUTS if step in compared else OUTS[:1]):
            out = out_tensor(w.batch, w.q_heads, w.head_dim, code)
            ol.ol_decode_step(ol.OL_LAYOUT_INT4, desc, dplanes[0], q_d, w.q_heads, kv_d, lens, lens_d, 0.0, -1, out,
                              code, ws, n)
            torch.cuda.synchronize()
            got[code] = out_as_f64(out)
        O.int4_append(*planes, kv, lens - 1)
        if step in compared:
            def row(b, q=q, kv=kv, lens=lens):
                sub = tuple(np.ascontiguousarray(p[:, b:b + 1]) for p in planes)
                return O.int4_attention(q[b:b + 1], *sub, lens[b:b + 1], cur_kv=np.ascontiguousarray(kv[:, b:b + 1]))[0]
            want = np.stack(threaded(row, list(range(w.batch))))
            for code, _ in OUTS:
                check(got[code], want, code)
        lens = lens + 1
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    for g, r in zip(dplanes, planes):
        np.testing.assert_array_equal(to_host(g), r)


def test_chunk4_full_size_sampled_rows():
    # the chunked step of bench.py: 4 tokens appended and attended per row, ragged rows of 512..8192
    w = WORKLOADS["chunk4_b32"]
    T = w.chunk
    case = make_case(w, history_len_offset=T)
    rng = np.random.default_rng(w.seed + 7)
    q = bf16_from_f32(rng.standard_normal((w.batch, w.q_heads, T, w.head_dim)).astype(np.float32))
    kv = bf16_from_f32(rng.standard_normal((2, w.batch, w.kv_heads, T, w.head_dim)).astype(np.float32))
    cache = contiguous_cache(case)
    case.history = None
    cache_d = to_dev(cache)
    desc = ol.kv_cache(cache_d, access=STABLE)
    n = ol.ol_workspace_size_chunk(w.batch, w.q_heads, w.kv_heads, w.head_dim, T)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    ol.ol_workspace_init(ws, n)
    q_d, kv_d, lens_d = to_dev(q), to_dev(kv), to_dev(case.lens)
    got = {}
    for code, dt in OUTS:
        out = torch.full((w.batch, w.q_heads, T, w.head_dim), float("nan"), dtype=dt, device="cuda")
        ol.ol_chunk_step(ol.OL_LAYOUT_CONTIGUOUS, desc, cache_d, q_d, w.q_heads, T, kv_d, case.lens, lens_d, 0.0, -1,
                         out, code, ws, n)
        torch.cuda.synchronize()
        got[code] = out_as_f64(out)
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    O.cache_update(cache, kv, case.lens - T)
    np.testing.assert_array_equal(to_host(cache_d), cache)    # every cache byte
    del cache_d
    rows = spread_rows(case.lens, extra=range(0, w.batch, 4))

    def row(b):
        return O.chunk_attention(q[b:b + 1], np.ascontiguousarray(cache[:, b:b + 1]), case.lens[b:b + 1], T)[0]
    want = np.stack(threaded(row, rows))
    for code, _ in OUTS:
        check(got[code][rows], want, code)


def test_hpaged_full_size_sampled_rows():
    # heterogeneous pages of bench.py: 64 rows over a pool of 65536 pages, each
    # page's formats chosen by its age; history appended by the oracle
    w = WORKLOADS["hpaged_b64"]
    case = make_case(w)
    S, M, H, D = w.page_size, w.max_pages_per_row, w.kv_heads, w.head_dim
    pool, desc = O.hpaged_pool(w.num_pages, H, S, D)
    table = block_table(case)
    cls = page_format_classes(case.lens, S, M)

    def fill(b):  # one append per run of pages of one format class; rows own disjoint pages
        h = case.history[b]
        hist, j = h.shape[2], 0
        npages = (hist + S - 1) // S
        while j < npages:
            j1 = j
            while j1 < npages and cls[b, j1] == cls[b, j]:
                j1 += 1
            kf, vf = AGE_FORMATS[cls[b, j]][1]
            O.hpaged_append(pool, desc, table[b:b + 1], h[:, None, :, j * S:min(j1 * S, hist)], [j * S],
                            O.page_desc(k=kf, v=vf))
            j = j1
    threaded(fill, list(range(w.batch)))
    case.history = None
    new_o = O.page_desc(*AGE_FORMATS[0][1])
    new_g = ol.page_format(*AGE_FORMATS[0][1])
    pool_d, fmt_d = to_dev(pool), to_dev(desc.view(np.uint8).copy())
    mirror = desc.copy().view(ol.PAGE_FORMAT_DTYPE)
    bt_d = to_dev(table)
    kvd = ol.hpaged_kv(pool_d, fmt_d, mirror, bt_d, table, kv_heads=H, page_size=S, head_dim=D, access=STABLE)
    ws, n = workspace(w.batch, w.q_heads, H, D)
    q_d, kv_d, lens_d = to_dev(case.q), to_dev(case.new_kv), to_dev(case.lens)
    got = {}
    for code, _ in OUTS:
        out = out_tensor(w.batch, w.q_heads, D, code)
        ol.ol_hpaged_decode_step(kvd, pool_d, q_d, w.q_heads, kv_d, new_g, case.lens, lens_d, 0.0, -1, out, code, ws,
                                 n)
        torch.cuda.synchronize()
        got[code] = out_as_f64(out)
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    rows = spread_rows(case.lens, extra=range(0, w.batch, 8))

    def row(b):
        return O.hpaged_attention(case.q[b:b + 1], pool, desc, table[b:b + 1], case.lens[b:b + 1], H,
                                  cur_kv=np.ascontiguousarray(case.new_kv[:, b:b + 1]))[0]
    want = np.stack(threaded(row, rows))                      # before the append: history only from the pages
    O.hpaged_append(pool, desc, table, case.new_kv, case.lens - 1, new_o)
    np.testing.assert_array_equal(to_host(fmt_d).view(np.uint8), desc.view(np.uint8))
    np.testing.assert_array_equal(mirror.view(np.uint8), desc.view(np.uint8))
    got_pool = to_host(pool_d)
    bad = np.argwhere(got_pool != pool)
    assert bad.size == 0, f"{len(bad)} pool bytes differ, first at page/byte {bad[0].tolist()}"
    for code, _ in OUTS:
        check(got[code][rows], want, code)


def test_int4_chunk4_full_size_sampled_rows():
    # the INT4 cache of 16 rows taking 4 tokens per row (bench.py's int4chunk4_b16):
    # attention on the tensor-core kernel with 2 query tokens per CTA (GQA 4), then
    # the quantized append; every plane byte compared, outputs on two rows
    w = WORKLOADS["int4chunk4_b16"]
    T = w.chunk
    case = make_case(w, history_len_offset=T)
    rng = np.random.default_rng(w.seed + 7)
    q = bf16_from_f32(rng.standard_normal((w.batch, w.q_heads, T, w.head_dim)).astype(np.float32))
    kv = bf16_from_f32(rng.standard_normal((2, w.batch, w.kv_heads, T, w.head_dim)).astype(np.float32))

    def quantized(b):
        sub = O.int4_planes(1, w.kv_heads, w.capacity, w.head_dim)
        O.int4_append(*sub, case.history[b][:, None], [0])
        return sub
    subs = threaded(quantized, list(range(w.batch)))
    planes = O.int4_planes(w.batch, w.kv_heads, w.capacity, w.head_dim)
    for b, sub in enumerate(subs):
        for full, part in zip(planes, sub):
            full[:, b] = part[:, 0]
    del subs
    case.history = None
    dplanes = tuple(to_dev(p) for p in planes)
    desc = ol.int4_kv(*dplanes, head_dim=w.head_dim, access=STABLE)
    n = ol.ol_workspace_size_chunk(w.batch, w.q_heads, w.kv_heads, w.head_dim, T)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    ol.ol_workspace_init(ws, n)
    q_d, kv_d, lens_d = to_dev(q), to_dev(kv), to_dev(case.lens)
    got = {}
    for code, dt in OUTS:
        out = torch.full((w.batch, w.q_heads, T, w.head_dim), float("nan"), dtype=dt, device="cuda")
        ol.ol_chunk_step(ol.OL_LAYOUT_INT4, desc, dplanes[0], q_d, w.q_heads, T, kv_d, case.lens, lens_d, 0.0, -1,
                         out, code, ws, n)
        torch.cuda.synchronize()
        got[code] = out_as_f64(out)
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    rows = [0, w.batch - 1]

    def row(b):
        sub = tuple(np.ascontiguousarray(p[:, b:b + 1]) for p in planes)
        return O.int4_chunk_attention(q[b:b + 1], *sub, case.lens[b:b + 1], T, np.ascontiguousarray(kv[:, b:b + 1]))[0]
    want = np.stack(threaded(row, rows))
    O.int4_append(*planes, kv, case.lens - T)
    for g, r in zip(dplanes, planes):
        np.testing.assert_array_equal(to_host(g), r)
    for code, _ in OUTS:
        check(got[code][rows], want, code)


def test_hpaged_chunk4_full_size_sampled_rows():
    # heterogeneous pages taking 4 tokens per row (bench.py's hpchunk4_b64): attention on the
    # tensor-core kernel with 2 query tokens per CTA, then the chunk encoded into its pages
    w = WORKLOADS["hpchunk4_b64"]
    T = w.chunk
    case = make_case(w, history_len_offset=T)
    rng = np.random.default_rng(w.seed + 7)
    q = bf16_from_f32(rng.standard_normal((w.batch, w.q_heads, T, w.head_dim)).astype(np.float32))
    kv = bf16_from_f32(rng.standard_normal((2, w.batch, w.kv_heads, T, w.head_dim)).astype(np.float32))
    S, M, H, D = w.page_size, w.max_pages_per_row, w.kv_heads, w.head_dim
    pool, desc = O.hpaged_pool(w.num_pages, H, S, D)
    table = block_table(case)
    cls = page_format_classes(case.lens, S, M)

    def fill(b):  # one append per run of pages of one format class; rows own disjoint pages
        h = case.history[b]
        hist, j = h.shape[2], 0
        npages = (hist + S - 1) // S
        while j < npages:
            j1 = j
            while j1 < npages and cls[b, j1] == cls[b, j]:
                j1 += 1
            kf, vf = AGE_FORMATS[cls[b, j]][1]
            O.hpaged_append(pool, desc, table[b:b + 1], h[:, None, :, j * S:min(j1 * S, hist)], [j * S],
                            O.page_desc(k=kf, v=vf))
            j = j1
    threaded(fill, list(range(w.batch)))
    case.history = None
    new_o = O.page_desc(*AGE_FORMATS[0][1])
    new_g = ol.page_format(*AGE_FORMATS[0][1])
    pool_d, fmt_d = to_dev(pool), to_dev(desc.view(np.uint8).copy())
    mirror = desc.copy().view(ol.PAGE_FORMAT_DTYPE)
    kvd = ol.hpaged_kv(pool_d, fmt_d, mirror, to_dev(table), table, kv_heads=H, page_size=S, head_dim=D,
                       access=STABLE)
    n = ol.ol_workspace_size_chunk(w.batch, w.q_heads, H, D, T)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    ol.ol_workspace_init(ws, n)
    q_d, kv_d, lens_d = to_dev(q), to_dev(kv), to_dev(case.lens)
    got = {}
    for code, dt in OUTS:
        out = torch.full((w.batch, w.q_heads, T, D), float("nan"), dtype=dt, device="cuda")
        ol.ol_hpaged_chunk_step(kvd, pool_d, q_d, w.q_heads, T, kv_d, new_g, case.lens, lens_d, 0.0, -1, out, code,
                                ws, n)
        torch.cuda.synchronize()
        got[code] = out_as_f64(out)
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    rows = [int(np.argmin(case.lens)), int(np.argmax(case.lens))]

    def row(b):
        return O.hpaged_chunk_attention(q[b:b + 1], pool, desc, table[b:b + 1], case.lens[b:b + 1], H, T,
                                        np.ascontiguousarray(kv[:, b:b + 1]))[0]
    want = np.stack(threaded(row, rows))                      # before the append: history only from the pages
    O.hpaged_append(pool, desc, table, kv, case.lens - T, new_o)
    np.testing.assert_array_equal(to_host(fmt_d).view(np.uint8), desc.view(np.uint8))
    got_pool = to_host(pool_d)
    bad = np.argwhere(got_pool != pool)
    assert bad.size == 0, f"{len(bad)} pool bytes differ, first at page/byte {bad[0].tolist()}"
    for code, _ in OUTS:
        check(got[code][rows], want, code)
