"""GPU parity of ol_decode_step_host: q, the new K/V, the lengths and y live in
host memory; the cache stays on the device. Mapped page-locked buffers are
read and written in place by the step's kernels; pageable or unaligned ones
go through the workspace with copies. Every mix must give the oracle's result
(cache bit-exact, outputs within 2e-3) exactly as the device-buffer call,
including batches whose lengths go to the device (more rows than the launch
carries by value)."""
import numpy as np
import pytest
import torch

import oracle as O
import place_kv_cache_gb300 as ol
from workloads import Workload, contiguous_cache, make_case
from tests.gpu_util import DEV, max_abs_err, to_dev, to_host

pytestmark = pytest.mark.gpu
TOL = 2e-3


def pinned(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def pinned_unaligned(a: np.ndarray) -> np.ndarray:
    """A page-locked copy of `a` starting 8 bytes past a 16-byte boundary."""
    a = np.ascontiguousarray(a)
    raw = torch.empty(a.nbytes + 64, dtype=torch.uint8).pin_memory().numpy()  # keeps the tensor alive
    off = (8 - raw.ctypes.data) % 16
    view = raw[off:off + a.nbytes].view(a.dtype).reshape(a.shape)
    np.copyto(view, a)
    assert view.ctypes.data % 16 == 8
    return view


# where each host buffer lives: (q, new K/V, y)
MEMORY = {
    "pinned": (pinned, pinned, pinned),
    "pageable": (np.ascontiguousarray, np.ascontiguousarray, np.ascontiguousarray),
    "mixed": (pinned, np.ascontiguousarray, pinned),
    "unaligned": (pinned_unaligned, pinned, pinned_unaligned),
}


def host_workspace(B, Hq, Hkv, D):
    n = ol.ol_workspace_size_host(B, Hq, Hkv, D)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    ol.ol_workspace_init(ws, n)
    return ws, n


@pytest.mark.parametrize("memory", ["pinned", "pageable", "mixed", "unaligned"])
@pytest.mark.parametrize("out_dtype", [ol.OL_F32, ol.OL_BF16], ids=["f32_out", "bf16_out"])
@pytest.mark.parametrize("shape", [
    ("gqa7", 1, 28, 4, 128, 1024, [513]),
    ("ragged", 5, 32, 8, 128, 600, [1, 16, 17, 599, 600]),
    ("many_rows", 200, 8, 2, 128, 64, None),     # lengths copied to the device
], ids=lambda s: s[0])
def test_host_step_contiguous(shape, out_dtype, memory):
    name, B, Hq, Hkv, D, C, lens = shape
    if name == "many_rows" and memory != "pinned":
        pytest.skip("the buffer kinds are covered by the smaller shapes")
    mq, mkv, mout = MEMORY[memory]
    w = Workload(name, "bf16", B, Hq, Hkv, D, C, "contiguous", seed=41, lens_range=(1, C))
    case = make_case(w, lens=None if lens is None else np.array(lens, np.int32))
    cache_np = contiguous_cache(case)
    cache_d = to_dev(cache_np)
    desc = ol.kv_cache(cache_d)
    ws, n = host_workspace(B, Hq, Hkv, D)
    out_h = mout(np.zeros((B, Hq, D), np.float32 if out_dtype == ol.OL_F32 else np.uint16))
    stream = torch.cuda.Stream()
    ol.ol_decode_step_host(ol.OL_LAYOUT_CONTIGUOUS, desc, cache_d, mq(case.q), Hq, mkv(case.new_kv),
                           case.lens, 0.0, -1, out_h, out_dtype, ws, n, stream=stream)
    stream.synchronize()
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    ref = cache_np.copy()
    O.cache_update(ref, case.new_kv, case.lens - 1)
    np.testing.assert_array_equal(to_host(cache_d), ref)
    want = O.decode_attention(case.q, ref, case.lens)
    got = out_h.numpy() if isinstance(out_h, torch.Tensor) else out_h
    got = got.astype(np.float64) if out_dtype == ol.OL_F32 else \
        (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    tol = TOL if out_dtype == ol.OL_F32 else TOL + 2.0 ** -8 * np.abs(want)
    assert np.all(np.abs(got - want) <= tol)


def test_host_step_int4():
    B, Hq, Hkv, D, C = 3, 16, 4, 128, 256
    w = Workload("h_i4", "bf16", B, Hq, Hkv, D, C, "int4", seed=42)
    case = make_case(w, lens=np.array([1, 100, 256], np.int32))
    planes = O.int4_planes(B, Hkv, C, D)
    for b, h in enumerate(case.history):
        if h.shape[2]:
            sub = O.int4_planes(1, Hkv, C, D)
            O.int4_append(*sub, h[:, None], [0])
            for full, part in zip(planes, sub):
                full[:, b] = part[:, 0]
    dplanes = tuple(to_dev(p) for p in planes)
    desc = ol.int4_kv(*dplanes, head_dim=D)
    ws, n = host_workspace(B, Hq, Hkv, D)
    out_h = pinned(np.zeros((B, Hq, D), np.float32))
    ol.ol_decode_step_host(ol.OL_LAYOUT_INT4, desc, dplanes[0], pinned(case.q), Hq, pinned(case.new_kv), case.lens,
                           0.0, -1, out_h, ol.OL_F32, ws, n)
    torch.cuda.synchronize()
    O.int4_append(*planes, case.new_kv, case.lens - 1)
    for g, r in zip((to_host(p) for p in dplanes), planes):
        np.testing.assert_array_equal(g, r)
    want = O.int4_attention(case.q, *planes, case.lens, cur_kv=case.new_kv)
    assert max_abs_err(out_h.numpy().astype(np.float64), want) <= TOL


def test_stats_describe_a_real_step():
    # the storage statistics of a step that ran on the GPU: no prefix copy, no
    # allocation, the appended bytes and the history bytes read
    B, Hq, Hkv, D, C = 2, 8, 2, 128, 64
    w = Workload("st", "bf16", B, Hq, Hkv, D, C, "contiguous", seed=43)
    case = make_case(w, lens=np.array([5, 64], np.int32))
    cache_d = to_dev(contiguous_cache(case))
    ws, n = host_workspace(B, Hq, Hkv, D)
    out_h = pinned(np.zeros((B, Hq, D), np.float32))
    ol.ol_reset_stats()
    ol.ol_decode_step_host(ol.OL_LAYOUT_CONTIGUOUS, ol.kv_cache(cache_d), cache_d, pinned(case.q), Hq,
                           pinned(case.new_kv), case.lens, 0.0, -1, out_h, ol.OL_F32, ws, n)
    torch.cuda.synchronize()
    s = ol.ol_last_call_stats()
    assert s["storage_prefix_copied_bytes"] == 0 and s["storage_allocations"] == 0
    assert s["storage_append_copied_bytes"] == 2 * B * Hkv * D * 2
    assert s["kv_payload_bytes_read"] == 2 * (4 + 63) * Hkv * D * 2
    assert ol.ol_total_stats()["calls"] == 1
