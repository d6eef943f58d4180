"""Parity at the full workload sizes, in the launch configuration bench.py
times (the default plan), against the CPU oracle: every output where the
oracle finishes in seconds, sampled rows elsewhere, and every cache byte.

Inputs follow the seeded recipe of each workload (workloads.WORKLOADS); the
cache history is laid out or quantized by the oracle-side helpers, never by
the CUDA path.
"""
import numpy as np
import pytest
import torch

import oracle as O
import place_kv_cache_gb300 as ol
from workloads import WORKLOADS, bf16_from_f32, block_table, contiguous_cache, make_case, poisoned_pool
from tests.gpu_util import check_out, out_as_f64, out_tensor, to_dev, to_host, workspace

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# the access bits bench.py gives its non-chained caches: history rows stable,
# so the first K/V tiles are requested before the dependency wait
STABLE = ol.OL_READ_WRITE | ol.OL_HISTORY_STABLE


def _pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def _step_contiguous(case, cache, host):
    w = case.workload
    cache_d = to_dev(cache)
    desc = ol.kv_cache(cache_d, access=STABLE)
    if host:  # the host-buffer call bench.py's e2e times: pinned q, new K/V and y used in place
        n = ol.ol_workspace_size_host(w.batch, w.q_heads, w.kv_heads, w.head_dim)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        ol.ol_workspace_init(ws, n)
        out = torch.full((w.batch, w.q_heads, w.head_dim), float("nan"), dtype=torch.bfloat16).pin_memory()
        ol.ol_decode_step_host(ol.OL_LAYOUT_CONTIGUOUS, desc, cache_d, _pinned(case.q), w.q_heads,
                               _pinned(case.new_kv), torch.from_numpy(case.lens), 0.0, -1, out, ol.OL_BF16, ws, n)
        torch.cuda.synchronize()
    else:
        ws, n = workspace(w.batch, w.q_heads, w.kv_heads, w.head_dim)
        out = out_tensor(w.batch, w.q_heads, w.head_dim, ol.OL_BF16)
        ol.ol_decode_step(ol.OL_LAYOUT_CONTIGUOUS, desc, cache_d, to_dev(case.q), w.q_heads, to_dev(case.new_kv),
                          case.lens, to_dev(case.lens), 0.0, -1, out, ol.OL_BF16, ws, n)
        torch.cuda.synchronize()
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    return cache_d, out_as_f64(out)


@pytest.mark.parametrize("host", [False, True], ids=["device_buffers", "host_buffers"])
@pytest.mark.parametrize("name", ["qwen_b1_gqa7", "ragged_b32"])
def test_contiguous_full_size(name, host):
    w = WORKLOADS[name]
    case = make_case(w)
    cache = contiguous_cache(case)
    cache_d, got = _step_contiguous(case, cache, host)
    O.cache_update(cache, case.new_kv, case.lens - 1)          # the expected cache, in place
    np.testing.assert_array_equal(to_host(cache_d), cache)
    del cache_d
    want = O.decode_attention(case.q, cache, case.lens)
    check_out(got, want, ol.OL_BF16)


def test_paged_full_size_sampled_rows():
    w = WORKLOADS["paged_b64"]
    case = make_case(w)
    table = block_table(case)
    pool = poisoned_pool(w)
    for b, h in enumerate(case.history):
        if h.shape[2]:
            O.paged_update(pool, table[b:b + 1], h[:, None], [0])
    case.history = None                                        # free the host copy of the history
    pool_d = to_dev(pool)
    bt_d = to_dev(table)
    ws, n = workspace(w.batch, w.q_heads, w.kv_heads, w.head_dim)
    out = out_tensor(w.batch, w.q_heads, w.head_dim, ol.OL_BF16)
    ol.ol_decode_step(ol.OL_LAYOUT_PAGED, ol.paged_kv(pool_d, bt_d, table, access=STABLE), pool_d, to_dev(case.q),
                      w.q_heads,
                      to_dev(case.new_kv), case.lens, to_dev(case.lens), 0.0, -1, out, ol.OL_BF16, ws, n)
    torch.cuda.synchronize()
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    got = out_as_f64(out)
    O.paged_update(pool, table, case.new_kv, case.lens - 1)
    np.testing.assert_array_equal(to_host(pool_d), pool)      # every pool byte
    del pool_d
    rows = sorted({int(np.argmin(case.lens)), int(np.argmax(case.lens)), 0, w.batch - 1, 17})
    want = O.paged_attention(case.q[rows], pool, table[rows], case.lens[rows])
    check_out(got[rows], want, ol.OL_BF16)


def test_int4_full_size_chained():
    # 64 chained steps at capacity 32768, history of 16384 tokens quantized by the oracle
    w = WORKLOADS["int4_b16"]
    case = make_case(w)
    planes = O.int4_planes(w.batch, w.kv_heads, w.capacity, w.head_dim)
    for b, h in enumerate(case.history):
        sub = O.int4_planes(1, w.kv_heads, w.capacity, w.head_dim)
        O.int4_append(*sub, h[:, None], [0])
        for full, part in zip(planes, sub):
            full[:, b] = part[:, 0]
    case.history = None
    dplanes = tuple(to_dev(p) for p in planes)
    desc = ol.int4_kv(*dplanes, head_dim=w.head_dim)
    ws, n = workspace(w.batch, w.q_heads, w.kv_heads, w.head_dim)
    rng = np.random.default_rng(w.seed + 1)
    lens = case.lens.copy()
    rows = [0, 7, w.batch - 1]
    for step in range(w.steps):
        q = bf16_from_f32(rng.standard_normal((w.batch, w.q_heads, w.head_dim)).astype(np.float32))
        kv = bf16_from_f32(rng.standard_normal((2, w.batch, w.kv_heads, 1, w.head_dim)).astype(np.float32))
        out = out_tensor(w.batch, w.q_heads, w.head_dim, ol.OL_BF16)
        ol.ol_decode_step(ol.OL_LAYOUT_INT4, desc, dplanes[0], to_dev(q), w.q_heads, to_dev(kv), lens, to_dev(lens),
                          0.0, -1, out, ol.OL_BF16, ws, n)
        torch.cuda.synchronize()
        O.int4_append(*planes, kv, lens - 1)
        if step in (0, 31, w.steps - 1):
            sub = tuple(np.ascontiguousarray(p[:, rows]) for p in planes)
            want = O.int4_attention(q[rows], *sub, lens[rows], cur_kv=np.ascontiguousarray(kv[:, rows]))
            check_out(out_as_f64(out)[rows], want, ol.OL_BF16)
        lens = lens + 1
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    for g, r in zip(dplanes, planes):
        np.testing.assert_array_equal(to_host(g), r)
