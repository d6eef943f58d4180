"""ol_decode_step_noalloc, the decode step for callers that cannot allocate
device memory (a host engine that owns all device memory and forbids
allocation while it executes, or a latency-critical loop that cannot take an
allocation's implicit synchronization): it must give what ol_decode_step gives
with a caller-provided workspace, on consecutive calls that reuse its static
scratch, and reject requests larger than that scratch before running anything.

This file is collected last so that a failure here leaves every other test run.
"""
import numpy as np
import pytest
import torch

import place_kv_cache_gb300 as ol
from workloads import Workload, bf16_from_f32, contiguous_cache, make_case
from tests.gpu_util import check_out, out_as_f64, out_tensor, to_dev, to_host, workspace

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_step_on_two_calls():
    w = Workload("noalloc", "bf16", 2, 28, 4, 128, 1024, "contiguous", seed=77)
    case = make_case(w, lens=np.array([700, 129], np.int32))
    cache = contiguous_cache(case)
    cache_ws, cache_na = to_dev(cache), to_dev(cache)
    desc_ws, desc_na = ol.kv_cache(cache_ws), ol.kv_cache(cache_na)
    ws, n = workspace(w.batch, w.q_heads, w.kv_heads, w.head_dim)
    rng = np.random.default_rng(78)
    lens = case.lens.copy()
    for call in range(2):
        q = to_dev(bf16_from_f32(rng.standard_normal((2, 28, 128)).astype(np.float32)))
        kv = to_dev(bf16_from_f32(rng.standard_normal((2, 2, 4, 1, 128)).astype(np.float32)))
        lens_d = to_dev(lens)
        out_ws = out_tensor(2, 28, 128, ol.OL_F32)
        out_na = out_tensor(2, 28, 128, ol.OL_F32)
        ol.ol_decode_step(ol.OL_LAYOUT_CONTIGUOUS, desc_ws, cache_ws, q, 28, kv, lens, lens_d, 0.0, -1, out_ws,
                          ol.OL_F32, ws, n)
        ol.ol_decode_step_noalloc(ol.OL_LAYOUT_CONTIGUOUS, desc_na, cache_na, q, 28, kv, lens, lens_d, 0.0, -1,
                                  out_na, ol.OL_F32)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_host(cache_na), to_host(cache_ws))
        check_out(out_as_f64(out_na), out_as_f64(out_ws), ol.OL_F32)
        lens = lens + 1


def test_noalloc_rejects_requests_beyond_its_scratch():
    # a batch whose worst-case workspace exceeds the static scratch: rejected before any launch
    batch, q_heads, kv_heads, head_dim = 4096, 8, 8, 128
    assert ol.ol_workspace_size(batch, q_heads, kv_heads, head_dim) > 16 * 1024 * 1024
    cache = torch.zeros(16, dtype=torch.bfloat16, device="cuda:0")
    desc = ol.kv_cache(cache, dims=(batch, kv_heads, 16, head_dim), dtype=ol.OL_BF16)
    q = torch.zeros(16, dtype=torch.bfloat16, device="cuda:0")
    before = cache.clone()
    with pytest.raises(ol.OlError) as e:
        ol.ol_decode_step_noalloc(ol.OL_LAYOUT_CONTIGUOUS, desc, cache, q, q_heads, q, np.ones(batch, np.int32), q,
                                  0.0, -1, q, ol.OL_F32)
    assert e.value.status == ol.OL_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.equal(cache, before)
