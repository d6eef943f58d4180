"""GPU parity of the chunked step (ol_chunk_step): new_len tokens appended per
row and attended causally inside the chunk, against the oracle (cache bytes
bit-exact, outputs within 2e-3). Covers the tensor-core kernel (head_dim 128,
GQA <= 8) and the CUDA-core kernel (fp32, head_dim 64, GQA 16), contiguous and
paged caches, chunk lengths 1..8, rows whose chunk is the whole row, finite
windows, and the chunk of one token against the decode step. INT4 caches: the
chunk attended uncompressed and quantized afterwards, codes / scales / zero
points bit-exact against the oracle's append."""
import zlib

import numpy as np
import pytest
import torch

import oracle as O
import place_kv_cache_gb300 as ol
from workloads import Workload, bf16_from_f32, block_table, contiguous_cache, make_case, poisoned_pool
from tests.gpu_util import DEV, max_abs_err, out_as_f64, out_tensor, to_dev, to_host

pytestmark = pytest.mark.gpu
TOL = 2e-3


def chunk_inputs(w, lens, T, seed):
    """History of lens - T tokens per row, and the chunk's q and K/V (seeded)."""
    case = make_case(w, lens=np.array(lens, np.int32), history_len_offset=T)
    rng = np.random.default_rng(seed)
    draw = lambda shape: rng.standard_normal(shape).astype(np.float32)  # noqa: E731
    store = (lambda a: bf16_from_f32(a)) if w.dtype == "bf16" else (lambda a: a)
    q = store(draw((w.batch, w.q_heads, T, w.head_dim)))
    kv = store(draw((2, w.batch, w.kv_heads, T, w.head_dim)))
    return case, q, kv


def ws_for(w, T):
    n = ol.ol_workspace_size_chunk(w.batch, w.q_heads, w.kv_heads, w.head_dim, T)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    ol.ol_workspace_init(ws, n)
    return ws, n


def out_for(w, T, out_dtype):
    return torch.empty((w.batch, w.q_heads, T, w.head_dim), device=DEV,
                       dtype=torch.float32 if out_dtype == ol.OL_F32 else torch.bfloat16)


CONTIG = [
    # name, dtype, B, Hq, Hkv, D, C, lens, T
    ("gqa7_t2", "bf16", 1, 28, 4, 128, 1024, [513], 2),
    ("ragged_t4", "bf16", 5, 32, 8, 128, 600, [4, 16, 17, 599, 600], 4),
    ("gqa2_t8", "bf16", 3, 4, 2, 128, 300, [8, 9, 300], 8),
    ("gqa16_generic_t3", "bf16", 2, 32, 2, 128, 200, [200, 77], 3),
    ("f32_d64_generic_t5", "f32", 2, 8, 2, 64, 160, [160, 5], 5),
]


@pytest.mark.parametrize("window", [-1, 0, 5, 40])
@pytest.mark.parametrize("shape", CONTIG, ids=lambda s: s[0])
def test_chunk_step_contiguous(shape, window):
    name, dt, B, Hq, Hkv, D, C, lens, T = shape
    w = Workload(name, dt, B, Hq, Hkv, D, C, "contiguous", seed=zlib.crc32(name.encode()) % 1000)
    case, q, kv = chunk_inputs(w, lens, T, seed=51)
    cache_np = contiguous_cache(case)
    cache_d = to_dev(cache_np)
    ptr0 = cache_d.data_ptr()
    ws, n = ws_for(w, T)
    out = out_for(w, T, ol.OL_F32)
    ol.ol_chunk_step(ol.OL_LAYOUT_CONTIGUOUS, ol.kv_cache(cache_d), cache_d, to_dev(q), Hq, T, to_dev(kv), case.lens,
                     to_dev(case.lens), 0.0, window, out, ol.OL_F32, ws, n)
    torch.cuda.synchronize()
    assert cache_d.data_ptr() == ptr0
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    ref = cache_np.copy()
    O.cache_update(ref, kv, case.lens - T)
    np.testing.assert_array_equal(to_host(cache_d), ref)
    want = O.chunk_attention(q, ref, case.lens, T, window=window)
    assert max_abs_err(out_as_f64(out), want) <= TOL


@pytest.mark.parametrize("window", [-1, 7])
def test_chunk_step_paged(window):
    name, B, Hq, Hkv, D, P, S, M, T = "pchunk", 4, 32, 8, 128, 128, 16, 16, 6
    w = Workload(name, "bf16", B, Hq, Hkv, D, M * S, "paged", seed=61, page_size=S, num_pages=P)
    case, q, kv = chunk_inputs(w, [6, 17, 100, 256], T, seed=52)
    pool = poisoned_pool(w)
    table = block_table(case)
    for b, h in enumerate(case.history):
        if h.shape[2]:
            O.paged_update(pool, table[b:b + 1], h[:, None], [0])
    pool_d = to_dev(pool)
    desc = ol.paged_kv(pool_d, to_dev(table), table)
    ws, n = ws_for(w, T)
    out = out_for(w, T, ol.OL_F32)
    ol.ol_chunk_step(ol.OL_LAYOUT_PAGED, desc, pool_d, to_dev(q), Hq, T, to_dev(kv), case.lens, to_dev(case.lens),
                     0.0, window, out, ol.OL_F32, ws, n)
    torch.cuda.synchronize()
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    ref = pool.copy()
    O.paged_update(ref, table, kv, case.lens - T)
    np.testing.assert_array_equal(to_host(pool_d), ref)
    want = O.paged_chunk_attention(q, ref, table, case.lens, T, window=window)
    assert max_abs_err(out_as_f64(out), want) <= TOL


def test_chunk_of_one_token_is_the_decode_step():
    w = Workload("one", "bf16", 3, 28, 4, 128, 512, "contiguous", seed=62)
    case = make_case(w, lens=np.array([1, 100, 512], np.int32))
    cache_np = contiguous_cache(case)
    outs = []
    for chunk in (True, False):
        cache_d = to_dev(cache_np)
        if chunk:
            ws, n = ws_for(w, 1)
            out = out_for(w, 1, ol.OL_F32)
            ol.ol_chunk_step(ol.OL_LAYOUT_CONTIGUOUS, ol.kv_cache(cache_d), cache_d, to_dev(case.q[:, :, None]), 28,
                             1, to_dev(case.new_kv), case.lens, to_dev(case.lens), 0.0, -1, out, ol.OL_F32, ws, n)
        else:
            n = ol.ol_workspace_size(3, 28, 4, 128)
            ws = torch.empty(n, dtype=torch.uint8, device=DEV)
            ol.ol_workspace_init(ws, n)
            out = out_tensor(3, 28, 128, ol.OL_F32)
            ol.ol_decode_step(ol.OL_LAYOUT_CONTIGUOUS, ol.kv_cache(cache_d), cache_d, to_dev(case.q), 28,
                              to_dev(case.new_kv), case.lens, to_dev(case.lens), 0.0, -1, out, ol.OL_F32, ws, n)
        torch.cuda.synchronize()
        outs.append((to_host(cache_d), out_as_f64(out).reshape(3, 28, 128)))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    # the decode step attends its new token from new_kv, the chunk from the cache it just
    # wrote: the same bf16 values, so the results agree to rounding
    assert np.abs(outs[0][1] - outs[1][1]).max() <= 1e-5


INT4 = [
    # name, B, Hq, Hkv, D, C, lens, T, quant mode (head_dim 128: tensor-core kernel, 8 / group query
    # tokens per CTA as MMA columns; head_dim 64: CUDA-core kernel)
    ("int4_gqa4_t4", 3, 16, 4, 128, 96, [4, 37, 96], 4, ol.OL_Q_DYNAMIC),
    ("int4_gqa7_t2_fixed", 1, 28, 4, 128, 64, [50], 2, ol.OL_Q_FIXED),
    ("int4_d64_t8", 2, 8, 2, 64, 48, [8, 48], 8, ol.OL_Q_DYNAMIC),
    ("int4_gqa4_t4_long", 3, 32, 8, 128, 2048, [5, 700, 2048], 4, ol.OL_Q_DYNAMIC),
    ("int4_gqa8_t3", 2, 16, 2, 128, 512, [300, 512], 3, ol.OL_Q_FIXED),
    ("int4_gqa2_t8", 2, 4, 2, 128, 272, [8, 200], 8, ol.OL_Q_DYNAMIC),
    ("int4_gqa1_t5_wide", 1, 6, 6, 128, 1024, [1000], 5, ol.OL_Q_DYNAMIC),
]


@pytest.mark.parametrize("window", [-1, 0, 9])
@pytest.mark.parametrize("shape", INT4, ids=lambda s: s[0])
def test_chunk_step_int4(shape, window):
    name, B, Hq, Hkv, D, C, lens, T, mode = shape
    w = Workload(name, "bf16", B, Hq, Hkv, D, C, "int4", seed=zlib.crc32(name.encode()) % 1000)
    case, q, kv = chunk_inputs(w, lens, T, seed=52)
    qm = dict(mode=O.Q_FIXED if mode == ol.OL_Q_FIXED else O.Q_DYNAMIC)
    planes = O.int4_planes(B, Hkv, C, D)
    for b, h in enumerate(case.history):
        if h.shape[2]:
            sub = O.int4_planes(1, Hkv, C, D)
            O.int4_append(*sub, h[:, None], [0], **qm)
            for full, part in zip(planes, sub):
                full[:, b] = part[:, 0]
    dev = [to_dev(a) for a in planes]
    desc = ol.int4_kv(dev[0], dev[1].view(torch.int16), dev[2], head_dim=D, quant_mode=mode)
    ws, n = ws_for(w, T)
    out = out_for(w, T, ol.OL_F32)
    ol.ol_chunk_step(ol.OL_LAYOUT_INT4, desc, dev[0], to_dev(q), Hq, T, to_dev(kv), case.lens, to_dev(case.lens), 0.0,
                     window, out, ol.OL_F32, ws, n)
    torch.cuda.synchronize()
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    want = O.int4_chunk_attention(q, *planes, case.lens, T, kv, window=window)
    assert max_abs_err(out_as_f64(out), want) <= TOL
    O.int4_append(*planes, kv, case.lens - T, **qm)
    for got, ref in zip(dev, planes):
        np.testing.assert_array_equal(to_host(got).view(ref.dtype), ref)
