"""GPU parity of the paged-cache path against the CPU oracle.

The pool is built by the oracle's PagedCacheUpdate from seeded history; the
CUDA step appends the new token through the block table and attends. Pool
bytes must be bit-exact (the new slot written, nothing else touched, unused
pages still NaN poison) and outputs within 2e-3 of the oracle.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle as O
import place_kv_cache_gb300 as ol
from workloads import Workload, block_table, make_case, poisoned_pool
from tests.gpu_util import check_out, max_abs_err, out_as_f64, out_tensor, to_dev, to_host, workspace

pytestmark = pytest.mark.gpu
TOL = 2e-3


def build_pool(case):
    """History of every row written through the block table by the oracle."""
    w = case.workload
    pool = poisoned_pool(w)
    table = block_table(case)
    for b, h in enumerate(case.history):
        if h.shape[2]:
            O.paged_update(pool, table[b:b + 1], h[:, None], [0])
    return pool, table


def paged_workload(name, dt, B, Hq, Hkv, D, P, S, M):
    return Workload(name, dt, B, Hq, Hkv, D, M * S, "paged", seed=zlib.crc32(name.encode()) % 1000,
                    page_size=S, num_pages=P, lens_range=(1, M * S))


def run(case, pool, table, out_dtype=ol.OL_F32, window=-1, step=True, flags=0):
    w = case.workload
    pool_d = to_dev(pool)
    ptr0 = pool_d.data_ptr()
    bt_d = to_dev(table)
    desc = ol.paged_kv(pool_d, bt_d, table, access=(ol.OL_READ_WRITE if step else ol.OL_READ_ONLY) | flags)
    ws, n = workspace(w.batch, w.q_heads, w.kv_heads, w.head_dim)
    out = out_tensor(w.batch, w.q_heads, w.head_dim, out_dtype)
    lens_d = to_dev(case.lens)
    if step:
        ol.ol_decode_step(ol.OL_LAYOUT_PAGED, desc, pool_d, to_dev(case.q), w.q_heads, to_dev(case.new_kv), case.lens,
                          lens_d, 0.0, window, out, out_dtype, ws, n)
    else:
        ol.ol_paged_decode_attention(desc, to_dev(case.q), w.q_heads, case.lens, lens_d, 0.0, window, out, out_dtype,
                                     ws, n)
    torch.cuda.synchronize()
    assert pool_d.data_ptr() == ptr0
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    return to_host(pool_d), out_as_f64(out)


SHAPES = [
    # name, dtype, B, Hq, Hkv, D, P, S, M, lens
    ("p16_gqa4", "bf16", 6, 32, 8, 128, 256, 16, 32, [1, 16, 17, 200, 511, 512]),
    ("p32_gqa7", "bf16", 2, 28, 4, 128, 64, 32, 16, [333, 512]),
    ("p64_gqa1", "bf16", 2, 2, 2, 128, 32, 64, 8, [64, 65]),
    ("p8_generic", "bf16", 3, 8, 2, 128, 128, 8, 32, [1, 100, 256]),
    ("p16_f32_d4", "f32", 2, 2, 1, 4, 16, 16, 4, [64, 3]),
    ("p16_gqa16_generic", "bf16", 2, 32, 2, 128, 64, 16, 16, [256, 30]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_paged_step_matches_oracle(shape):
    name, dt, B, Hq, Hkv, D, P, S, M, lens = shape
    w = paged_workload(name, dt, B, Hq, Hkv, D, P, S, M)
    case = make_case(w, lens=np.array(lens, np.int32))
    pool, table = build_pool(case)
    got_pool, got = run(case, pool, table)
    ref = pool.copy()
    O.paged_update(ref, table, case.new_kv, case.lens - 1)
    want = O.paged_attention(case.q, ref, table, case.lens)
    np.testing.assert_array_equal(got_pool.view(np.uint8), ref.view(np.uint8))
    assert max_abs_err(got, want) <= TOL, max_abs_err(got, want)


@pytest.mark.parametrize("window", [0, 1, 16, 100])
def test_paged_attention_window_read_only(window):
    w = paged_workload("pw", "bf16", 4, 32, 8, 128, 256, 16, 32)
    case = make_case(w, lens=np.array([5, 16, 300, 512], np.int32), history_len_offset=0)
    pool, table = build_pool(case)
    got_pool, got = run(case, pool, table, window=window, step=False, out_dtype=ol.OL_BF16)
    np.testing.assert_array_equal(got_pool.view(np.uint8), pool.view(np.uint8))
    want = O.paged_attention(case.q, pool, table, case.lens, window=window)
    check_out(got, want, ol.OL_BF16)


def test_paged_equals_contiguous_on_gpu():
    # the same logical cache through a random block table and as a contiguous cache
    w = paged_workload("pc", "bf16", 3, 16, 4, 128, 128, 16, 16)
    case = make_case(w, lens=np.array([256, 97, 1], np.int32), history_len_offset=0)
    pool, table = build_pool(case)
    _, got_paged = run(case, pool, table, step=False)
    from workloads import contiguous_cache
    cache = contiguous_cache(case)
    cache_d = to_dev(cache)
    ws, n = workspace(3, 16, 4, 128)
    out = out_tensor(3, 16, 128, ol.OL_F32)
    ol.ol_decode_attention(ol.kv_cache(cache_d, access=ol.OL_READ_ONLY), to_dev(case.q), 16, case.lens,
                           to_dev(case.lens), 0.0, -1, out, ol.OL_F32, ws, n)
    torch.cuda.synchronize()
    got_contig = out_as_f64(out)
    assert max_abs_err(got_paged, got_contig) <= 1e-6


def test_paged_cache_update_standalone():
    w = paged_workload("pu", "bf16", 3, 4, 2, 128, 64, 16, 8)
    case = make_case(w, lens=np.array([40, 3, 100], np.int32))
    pool, table = build_pool(case)
    rng = np.random.default_rng(3)
    from workloads import bf16_from_f32
    vals = bf16_from_f32(rng.standard_normal((2, 3, 2, 3, 128)).astype(np.float32))
    pos = np.array([39, 2, 99], np.int32)
    pool_d = to_dev(pool)
    desc = ol.paged_kv(pool_d, to_dev(table), table)
    ol.ol_paged_cache_update(desc, pool_d, to_dev(vals), 3, pos, to_dev(pos))
    torch.cuda.synchronize()
    ref = pool.copy()
    O.paged_update(ref, table, vals, pos)
    np.testing.assert_array_equal(to_host(pool_d).view(np.uint8), ref.view(np.uint8))


def test_paged_history_stable_flag():
    name, dt, B, Hq, Hkv, D, P, S, M, lens = SHAPES[0]
    w = paged_workload(name, dt, B, Hq, Hkv, D, P, S, M)
    case = make_case(w, lens=np.array(lens, np.int32))
    pool, table = build_pool(case)
    got_pool, got = run(case, pool, table, flags=ol.OL_HISTORY_STABLE)
    ref = pool.copy()
    O.paged_update(ref, table, case.new_kv, case.lens - 1)
    np.testing.assert_array_equal(got_pool.view(np.uint8), ref.view(np.uint8))
    check_out(got, O.paged_attention(case.q, ref, table, case.lens), ol.OL_F32)
