"""GPU parity of the contiguous-cache path against the CPU oracle.

Bar: cache bytes bit-exact after every append; attention outputs within a
max-abs error of 2e-3 of the fp64 oracle (bf16 inputs, fp32 accumulation).
Cases span several 16-token tiles, ragged tails, capacities that are not a
multiple of 16, lengths 1 / 16 / 17 / capacity, GQA groups 1..16, head_dim
4..256, fp32 and bf16 caches, bf16 and fp32 outputs and finite windows.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle as O
import place_kv_cache_gb300 as ol
from workloads import WORKLOADS, Workload, contiguous_cache, make_case
from tests.gpu_util import (canaries_intact, check_out, guarded, max_abs_err, out_as_f64, out_tensor, place,
                            to_dev, to_host, workspace)

pytestmark = pytest.mark.gpu
TOL = 2e-3


def run_step(case, cache_np, out_dtype=ol.OL_F32, window=-1, scale=0.0, access=ol.OL_READ_WRITE):
    w = case.workload
    cache_d = to_dev(cache_np)
    ptr0 = cache_d.data_ptr()
    desc = ol.kv_cache(cache_d, access=access)
    ws, n = workspace(w.batch, w.q_heads, w.kv_heads, w.head_dim)
    out = out_tensor(w.batch, w.q_heads, w.head_dim, out_dtype)
    lens_d = to_dev(case.lens)
    ol.ol_decode_step(ol.OL_LAYOUT_CONTIGUOUS, desc, cache_d, to_dev(case.q), w.q_heads, to_dev(case.new_kv),
                      case.lens, lens_d, scale, window, out, out_dtype, ws, n)
    torch.cuda.synchronize()
    assert cache_d.data_ptr() == ptr0
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    return to_host(cache_d), out_as_f64(out)


def expected(case, cache_np, window=-1, scale=None):
    ref = cache_np.copy()
    O.cache_update(ref, case.new_kv, case.lens - 1)
    return ref, O.decode_attention(case.q, ref, case.lens, scale=scale, window=window)


SHAPES = [
    # name, dtype, B, Hq, Hkv, D, C, lens
    ("gqa7", "bf16", 1, 28, 4, 128, 1024, [513]),
    ("ragged", "bf16", 5, 32, 8, 128, 600, [1, 16, 17, 599, 600]),
    ("gqa1", "bf16", 3, 2, 2, 128, 96, [33, 96, 1]),
    ("gqa8", "bf16", 2, 16, 2, 128, 300, [257, 129]),
    ("gqa16_generic", "bf16", 2, 32, 2, 128, 200, [200, 77]),
    ("d64_generic", "bf16", 2, 8, 2, 64, 160, [160, 5]),
    ("d256_generic", "bf16", 1, 4, 1, 256, 80, [80]),
    ("f32_d128_generic", "f32", 2, 8, 2, 128, 128, [128, 40]),
    ("f32_d4", "f32", 2, 3, 1, 4, 16, [16, 9]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("out_dtype", [ol.OL_F32, ol.OL_BF16], ids=["out_f32", "out_bf16"])
def test_step_matches_oracle(shape, out_dtype):
    name, dt, B, Hq, Hkv, D, C, lens = shape
    w = Workload(name, dt, B, Hq, Hkv, D, C, "contiguous", seed=zlib.crc32(name.encode()) % 1000)
    case = make_case(w, lens=np.array(lens, np.int32))
    cache = contiguous_cache(case)
    got_cache, got = run_step(case, cache, out_dtype)
    ref_cache, want = expected(case, cache)
    np.testing.assert_array_equal(got_cache.view(np.uint8), ref_cache.view(np.uint8))
    check_out(got, want, out_dtype)


@pytest.mark.parametrize("window", [0, 1, 15, 16, 33, 5000])
def test_step_with_window(window):
    w = Workload("win", "bf16", 4, 16, 4, 128, 640, "contiguous", seed=7)
    case = make_case(w, lens=np.array([1, 17, 300, 640], np.int32))
    cache = contiguous_cache(case)
    _, got = run_step(case, cache, window=window)
    _, want = expected(case, cache, window=window)
    assert max_abs_err(got, want) <= TOL


def test_explicit_scale():
    w = Workload("scale", "bf16", 2, 8, 2, 128, 256, "contiguous", seed=8)
    case = make_case(w, lens=np.array([200, 31], np.int32))
    cache = contiguous_cache(case)
    _, got = run_step(case, cache, scale=0.3)
    _, want = expected(case, cache, scale=0.3)
    assert max_abs_err(got, want) <= TOL


@pytest.mark.parametrize("dt,D", [("bf16", 128), ("f32", 4), ("bf16", 64)])
def test_attention_only_reads_and_never_writes(dt, D):
    # ol_decode_attention on a READ_ONLY descriptor: y matches the oracle, the cache is untouched,
    # including rows with nothing to attend (lens 0 -> y = 0)
    w = Workload("ro", dt, 3, 8, 2, D, 200, "contiguous", seed=9)
    case = make_case(w, lens=np.array([0, 200, 45], np.int32), history_len_offset=0)
    cache = contiguous_cache(case)
    cache_d = to_dev(cache)
    desc = ol.kv_cache(cache_d, access=ol.OL_READ_ONLY)
    ws, n = workspace(w.batch, w.q_heads, w.kv_heads, D)
    out = out_tensor(w.batch, w.q_heads, D, ol.OL_F32)
    ol.ol_decode_attention(desc, to_dev(case.q), w.q_heads, case.lens, to_dev(case.lens), 0.0, -1, out, ol.OL_F32,
                           ws, n)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(cache_d).view(np.uint8), cache.view(np.uint8))
    want = O.decode_attention(case.q, cache, case.lens)
    got = out_as_f64(out)
    assert max_abs_err(got, want) <= TOL
    np.testing.assert_array_equal(got[0], 0.0)


def test_cache_update_rows_and_scalar():
    w = Workload("upd", "bf16", 3, 4, 2, 128, 64, "contiguous", seed=10)
    rng = np.random.default_rng(10)
    cache = (rng.standard_normal((2, 3, 2, 64, 128)).astype(np.float32))
    from workloads import bf16_from_f32
    cache = bf16_from_f32(cache)
    vals = bf16_from_f32(rng.standard_normal((2, 3, 2, 5, 128)).astype(np.float32))
    buf, payload = guarded(cache.nbytes)
    cache_d = place(payload, cache)
    desc = ol.kv_cache(cache_d)
    pos = np.array([0, 30, 59], np.int32)
    ol.ol_cache_update_rows(desc, cache_d, to_dev(vals), 5, pos, to_dev(pos))
    torch.cuda.synchronize()
    ref = cache.copy()
    O.cache_update(ref, vals, pos)
    np.testing.assert_array_equal(to_host(cache_d), ref)
    ol.ol_cache_update(desc, cache_d, to_dev(vals), 5, 11)
    torch.cuda.synchronize()
    O.cache_update(ref, vals, np.array([11, 11, 11], np.int32))
    np.testing.assert_array_equal(to_host(cache_d), ref)
    assert canaries_intact(buf)
    with pytest.raises(ol.OlError) as e:
        ol.ol_cache_update(desc, cache_d, to_dev(vals), 5, 60)
    assert e.value.status == ol.OL_ERR_CAPACITY


def test_tiny_f32_four_chained_steps():
    # the 4-step fp32 fixture: append at position t, attend t + 1 tokens, pointer identity every step
    w = WORKLOADS["tiny_f32"]
    rng = np.random.default_rng(w.seed)
    cache = np.full((2, 1, 1, w.capacity, w.head_dim), np.nan, np.float32)
    cache_d = to_dev(cache)
    ptr0 = cache_d.data_ptr()
    desc = ol.kv_cache(cache_d)
    ws, n = workspace(1, 1, 1, w.head_dim)
    ref = cache.copy()
    for t in range(w.steps):
        q = rng.uniform(-1, 1, (1, 1, w.head_dim)).astype(np.float32)
        kv = rng.uniform(-1, 1, (2, 1, 1, 1, w.head_dim)).astype(np.float32)
        lens = np.array([t + 1], np.int32)
        out = out_tensor(1, 1, w.head_dim, ol.OL_F32)
        ol.ol_decode_step(ol.OL_LAYOUT_CONTIGUOUS, desc, cache_d, to_dev(q), 1, to_dev(kv), lens, to_dev(lens), 0.0,
                          -1, out, ol.OL_F32, ws, n)
        torch.cuda.synchronize()
        assert cache_d.data_ptr() == ptr0
        O.cache_update(ref, kv, [t])
        want = O.decode_attention(q, ref, lens)
        np.testing.assert_array_equal(to_host(cache_d).view(np.uint32), ref.view(np.uint32))
        assert max_abs_err(out_as_f64(out), want) <= 1e-5


def test_fault_injection_leaves_cache_untouched(monkeypatch):
    w = Workload("inj", "bf16", 2, 8, 2, 128, 64, "contiguous", seed=11)
    case = make_case(w, lens=np.array([10, 64], np.int32))
    cache = contiguous_cache(case)
    cache_d = to_dev(cache)
    ws, n = workspace(2, 8, 2, 128)
    out = out_tensor(2, 8, 128, ol.OL_F32)
    monkeypatch.setenv("OL_FAULT_INJECT", "after_validate")
    with pytest.raises(ol.OlError) as e:
        ol.ol_decode_step(ol.OL_LAYOUT_CONTIGUOUS, ol.kv_cache(cache_d), cache_d, to_dev(case.q), 8,
                          to_dev(case.new_kv), case.lens, to_dev(case.lens), 0.0, -1, out, ol.OL_F32, ws, n)
    assert e.value.status == ol.OL_ERR_INJECTED
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(cache_d).view(np.uint8), cache.view(np.uint8))
    assert torch.isnan(out).all()


@pytest.mark.parametrize("shape", [SHAPES[0], SHAPES[1], SHAPES[4], SHAPES[8]], ids=lambda s: s[0])
def test_history_stable_flag_gives_the_same_step(shape):
    # the caller's promise that the history is stable only moves the first tile
    # requests before the dependency wait; results are those of a plain step
    name, dt, B, Hq, Hkv, D, C, lens = shape
    w = Workload(name, dt, B, Hq, Hkv, D, C, "contiguous", seed=zlib.crc32(name.encode()) % 1000)
    case = make_case(w, lens=np.array(lens, np.int32))
    cache = contiguous_cache(case)
    got_cache, got = run_step(case, cache, access=ol.OL_READ_WRITE | ol.OL_HISTORY_STABLE)
    ref_cache, want = expected(case, cache)
    np.testing.assert_array_equal(got_cache.view(np.uint8), ref_cache.view(np.uint8))
    check_out(got, want, ol.OL_F32)


def test_large_batch_reads_lengths_from_device():
    # more than 160 rows: the kernels map CTAs from lens_dev rather than from the launch
    rng = np.random.default_rng(21)
    lens = rng.integers(1, 65, size=200).astype(np.int32)
    w = Workload("bigb", "bf16", 200, 8, 2, 128, 64, "contiguous", seed=21)
    case = make_case(w, lens=lens)
    cache = contiguous_cache(case)
    got_cache, got = run_step(case, cache)
    ref_cache, want = expected(case, cache)
    np.testing.assert_array_equal(got_cache.view(np.uint8), ref_cache.view(np.uint8))
    check_out(got, want, ol.OL_F32)
