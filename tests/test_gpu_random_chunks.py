"""Seeded random sweeps of chunked steps (several new tokens per row, causal
attention inside the chunk) on the GPU against the CPU oracle, for the INT4
cache and the heterogeneous paged cache: drawn batch, kv heads, query group
(1-8: one or two query tokens per MMA column group, odd and even numbers of
slices, a single slice), chunk length, lengths (a row with no history and a
full row included), windows and quantization mode or page formats. The
planner picks the split plan per shape, so the sweep reaches combinations of
column groups, splits and windows the hand-picked shapes do not. The cache
must match the oracle's append byte for byte and every output the oracle's
attention within 2e-3.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle as O
import place_kv_cache_gb300 as ol
from workloads import Workload, bf16_from_f32
from tests.gpu_util import check_out, max_abs_err, out_as_f64, to_dev, to_host
from tests.test_gpu_chunk import TOL, chunk_inputs, out_for, ws_for
from tests.test_gpu_hpaged import FORMATS, Pair, fmt_pair

pytestmark = pytest.mark.gpu


def draw_int4_chunks(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        B = int(rng.integers(1, 5))
        Hkv = int(rng.integers(1, 5))
        G = int(rng.integers(1, 9))
        D = 128 if rng.random() < 0.85 else 64
        C = 16 * int(rng.integers(2, 65))
        T = int(rng.integers(2, 10))
        lens = rng.integers(T, C + 1, size=B)
        if B > 1:  # edge rows: no history, and a full row
            lens[int(rng.integers(B))] = T
            lens[int(rng.integers(B))] = C
        window = int(rng.choice([-1, -1, 0, 3, 40]))
        mode = ol.OL_Q_FIXED if rng.integers(2) else ol.OL_Q_DYNAMIC
        cases.append(dict(id=f"{i:02d}-B{B}-H{Hkv}x{G}-D{D}-C{C}-T{T}-w{window}-{'fixed' if mode == ol.OL_Q_FIXED else 'dyn'}",
                          B=B, Hkv=Hkv, G=G, D=D, C=C, T=T, lens=lens.astype(np.int32), window=window, mode=mode))
    return cases


INT4_CHUNKS = draw_int4_chunks(16, 2029)


@pytest.mark.parametrize("c", INT4_CHUNKS, ids=[c["id"] for c in INT4_CHUNKS])
def test_random_int4_chunk_step(c):
    B, Hkv, G, D, C, T, window, mode = c["B"], c["Hkv"], c["G"], c["D"], c["C"], c["T"], c["window"], c["mode"]
    Hq = Hkv * G
    w = Workload("rc_" + c["id"], "bf16", B, Hq, Hkv, D, C, "int4", seed=zlib.crc32(c["id"].encode()) % 1000)
    case, q, kv = chunk_inputs(w, c["lens"], T, seed=zlib.crc32(c["id"].encode()) % 997)
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


def draw_hpaged_chunks(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        B = int(rng.integers(1, 4))
        H = int(rng.integers(1, 4))
        S = int(rng.choice([16, 32]))
        G = int(rng.integers(1, 9))
        T = int(rng.integers(2, 10))
        hist = rng.integers(0, 400, size=B)
        if B > 1:
            hist[int(rng.integers(B))] = 0  # a row whose chunk starts at slot 0
        window = int(rng.choice([-1, -1, 0, 5]))
        cases.append(dict(id=f"{i:02d}-B{B}-H{H}x{G}-S{S}-T{T}-w{window}", B=B, H=H, S=S, G=G, T=T,
                          hist=hist.astype(np.int32), window=window, fmt_seed=int(rng.integers(1 << 30))))
    return cases


HPAGED_CHUNKS = draw_hpaged_chunks(12, 2030)


@pytest.mark.parametrize("c", HPAGED_CHUNKS, ids=[c["id"] for c in HPAGED_CHUNKS])
def test_random_hpaged_chunk_step(c):
    B, H, S, G, T, hist, window = c["B"], c["H"], c["S"], c["G"], c["T"], c["hist"], c["window"]
    D, Hq = 128, H * G
    M = int(-(-(int(hist.max()) + T) // S)) + 1
    pr = Pair(B, H, S, D, M, B * M + 1, seed=zlib.crc32(c["id"].encode()) % 10007)
    frng = np.random.default_rng(c["fmt_seed"])
    fmts = frng.integers(0, len(FORMATS), size=(B, M))
    pr.fill(hist, lambda b, j: int(fmts[b, j]))
    lens = hist + T
    q = bf16_from_f32(pr.rng.standard_normal((B, Hq, T, D)).astype(np.float32))
    new_kv = pr.values(T)
    od, gd = fmt_pair(int(frng.integers(len(FORMATS))))
    want = O.hpaged_chunk_attention(q, pr.pool, pr.desc, pr.table, lens, H, T, new_kv, window=window)
    O.hpaged_append(pr.pool, pr.desc, pr.table, new_kv, hist, od)
    n = ol.ol_workspace_size_chunk(B, Hq, H, D, T)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda:0")
    ol.ol_workspace_init(ws, n)
    out = torch.full((B, Hq, T, D), float("nan"), dtype=torch.float32, device="cuda:0")
    ol.ol_hpaged_chunk_step(pr.kv, pr.pool_d, to_dev(q), Hq, T, to_dev(new_kv), gd, lens, to_dev(lens), 0.0, window,
                            out, ol.OL_F32, ws, n)
    torch.cuda.synchronize()
    check_out(out_as_f64(out), want, ol.OL_F32)
    pr.check_state()
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
