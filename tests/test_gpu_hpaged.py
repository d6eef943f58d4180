"""GPU parity of the heterogeneous paged cache (per-page K/V formats) against
the CPU oracle.

Both sides run the same sequence of calls on the same seeded values: appends
that start, continue and fill pages with changing formats, fused decode steps,
selected-page conversion. After every call the pool bytes, the device format
table and the host mirror must equal the oracle's bit for bit (bytes the
method never writes keep their 0xA5 fill); attention outputs are within 2e-3
of the oracle's fp64 result (plus half a bf16 ulp for bf16 outputs).
"""
import numpy as np
import pytest
import torch

import oracle as O
import place_kv_cache_gb300 as ol
from workloads import bf16_from_f32
from tests.gpu_util import check_out, out_as_f64, out_tensor, to_dev, to_host, workspace

pytestmark = pytest.mark.gpu

# (format, scale, zero point) pairs for K and V, covering every format
FORMATS = [
    ((O.HF_BF16, 1.0, 0), (O.HF_BF16, 1.0, 0)),
    ((O.HF_I8, 0.03125, 0), (O.HF_U4, 0.5, 8)),
    ((O.HF_F32, 1.0, 0), (O.HF_I2, 0.8, 0)),
    ((O.HF_F16, 1.0, 0), (O.HF_U8, 0.025, 128)),
    ((O.HF_I4, 0.45, 0), (O.HF_U2, 0.9, 2)),
    ((O.HF_U4, 0.5, 7), (O.HF_F16, 1.0, 0)),
    ((O.HF_I8, 0.02, -5), (O.HF_F32, 1.0, 0)),
    ((O.HF_U2, 0.7, 1), (O.HF_I4, 0.3, -1)),
]


def fmt_pair(i):
    k, v = FORMATS[i % len(FORMATS)]
    return O.page_desc(k=k, v=v), ol.page_format(k=k, v=v)


class Pair:
    """The oracle's cache state and the device's, built by the same calls."""

    def __init__(self, B, H, S, D, M, P, seed):
        self.rng = np.random.default_rng(seed)
        self.B, self.H, self.S, self.D, self.M, self.P = B, H, S, D, M, P
        self.table = self.rng.permutation(P)[: B * M].astype(np.int32).reshape(B, M)
        self.pool, self.desc = O.hpaged_pool(P, H, S, D)
        self.pool[:] = 0xA5
        self.pool_d = to_dev(self.pool.copy())
        self.fmt_d = to_dev(self.desc.view(np.uint8).copy())
        self.mirror = self.desc.copy().view(ol.PAGE_FORMAT_DTYPE)
        self.bt_d = to_dev(self.table)
        self.kv = ol.hpaged_kv(self.pool_d, self.fmt_d, self.mirror, self.bt_d, self.table, kv_heads=H, page_size=S,
                               head_dim=D)

    def values(self, n, lead=2, std=1.5):
        x = self.rng.standard_normal((lead, self.B, self.H, n, self.D)).astype(np.float32) * np.float32(std)
        return bf16_from_f32(x)

    def append(self, pos, vals, fi):
        od, gd = fmt_pair(fi)
        pos = np.asarray(pos, np.int32)
        O.hpaged_append(self.pool, self.desc, self.table, vals, pos, od)
        vals_d = to_dev(vals) if vals.size else to_dev(np.zeros(8, np.uint16))   # an empty tensor has no address
        ol.ol_hpaged_append(self.kv, self.pool_d, vals_d, vals.shape[3], pos, to_dev(pos), gd)

    def check_state(self):
        torch.cuda.synchronize()
        got = to_host(self.pool_d)
        bad = np.argwhere(got != self.pool)
        assert bad.size == 0, f"{len(bad)} pool bytes differ, first at page/byte {bad[0].tolist()}"
        np.testing.assert_array_equal(to_host(self.fmt_d).view(np.uint8), self.desc.view(np.uint8))
        np.testing.assert_array_equal(self.mirror.view(np.uint8), self.desc.view(np.uint8))

    def fill(self, lens, fmt_of_page=lambda b, j: j):
        """History of every row, page by page, page j of row b started in formats fmt_of_page(b, j)
        (one row per call: the pages one call starts share its formats)."""
        for j in range(self.M):
            for b in range(self.B):
                n = min(self.S, int(lens[b]) - j * self.S)
                if n > 0:
                    self._append_row(b, j * self.S, self.values(n, lead=2)[:, b:b + 1], fmt_of_page(b, j))

    def _append_row(self, b, pos, vals, fi):
        od, gd = fmt_pair(fi)
        t = np.ascontiguousarray(self.table[b:b + 1])
        p = np.array([pos], np.int32)
        O.hpaged_append(self.pool, self.desc, t, vals, p, od)
        kv = ol.hpaged_kv(self.pool_d, self.fmt_d, self.mirror, to_dev(t), t, kv_heads=self.H, page_size=self.S,
                          head_dim=self.D)
        ol.ol_hpaged_append(kv, self.pool_d, to_dev(vals), vals.shape[3], p, to_dev(p), gd)


APPEND_SHAPES = [
    # B, H, S, D, M
    (3, 2, 16, 128, 6),
    (2, 1, 4, 4, 8),
    (2, 4, 8, 64, 5),
    (1, 2, 16, 256, 3),
]


@pytest.mark.parametrize("shape", APPEND_SHAPES, ids=[f"b{s[0]}h{s[1]}s{s[2]}d{s[3]}" for s in APPEND_SHAPES])
def test_append_sequence_matches_oracle(shape):
    B, H, S, D, M = shape
    pr = Pair(B, H, S, D, M, B * M + 3, seed=101 + D)
    pos = np.array([(b * 5) % S for b in range(B)], np.int32)     # row 0 starts page 0; others continue it
    for i, n in enumerate([2 * S + 3, 1, S, 3, 0, S - 1, 2]):
        n = min(n, M * S - int(pos.max()))
        pr.append(pos, pr.values(n), i)
        pr.check_state()
        pos = pos + n


GQA = [  # B, H, S, D, Hq
    (1, 2, 16, 128, 8), (2, 2, 16, 128, 14), (3, 1, 8, 64, 16), (2, 2, 4, 4, 4), (1, 2, 16, 256, 32),
    # tensor-core kernel: groups 1-3 (duplicated columns with dead ones), 5 and 8 (P^T hi and lo apart)
    (1, 4, 16, 128, 4), (1, 2, 16, 128, 4), (2, 2, 16, 128, 6), (1, 2, 16, 128, 10), (1, 1, 16, 128, 8)]


@pytest.mark.parametrize("shape", GQA, ids=[f"b{s[0]}h{s[1]}s{s[2]}d{s[3]}g{s[4] // s[1]}" for s in GQA])
@pytest.mark.parametrize("out_dtype", [ol.OL_F32, ol.OL_BF16])
def test_attention_over_mixed_pages_matches_oracle(shape, out_dtype):
    B, H, S, D, Hq = shape
    M = 12
    pr = Pair(B, H, S, D, M, B * M, seed=202 + Hq)
    lens = np.array([M * S - 3 * b - (b == 1) * 40 for b in range(B)], np.int32)
    lens = np.clip(lens, 1, M * S)
    pr.fill(lens, lambda b, j: j + b)
    pr.check_state()
    q = bf16_from_f32(pr.rng.standard_normal((B, Hq, D)).astype(np.float32))
    cur = pr.values(1)
    ws, n = workspace(B, Hq, H, D)
    for cur_kv in (None, cur):
        for window in (-1, 0, S + 1, 5 * S - 2):
            out = out_tensor(B, Hq, D, out_dtype)
            ol.ol_hpaged_decode_attention(pr.kv, to_dev(q), Hq, lens, to_dev(lens),
                                          None if cur_kv is None else to_dev(cur_kv), 0.0, window, out, out_dtype,
                                          ws, n)
            torch.cuda.synchronize()
            want = O.hpaged_attention(q, pr.pool, pr.desc, pr.table, lens, H, cur_kv=cur_kv, window=window)
            check_out(out_as_f64(out), want, out_dtype)
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    pr.check_state()   # attention wrote nothing


@pytest.mark.parametrize("shape", [(3, 2, 16, 128, 8), (2, 1, 4, 8, 4)], ids=["s16d128g4", "s4d8g4"])
def test_fused_steps_match_oracle(shape):
    B, H, S, D, Hq = shape
    M = 6
    pr = Pair(B, H, S, D, M, B * M + 1, seed=303 + D)
    lens = np.array([S - 2 + b for b in range(B)], np.int32)        # steps cross page boundaries
    pr.fill(lens - 1, lambda b, j: 3 * j + b)
    ws, n = workspace(B, Hq, H, D)
    for i in range(6):
        q = bf16_from_f32(pr.rng.standard_normal((B, Hq, D)).astype(np.float32))
        new_kv = pr.values(1)
        od, gd = fmt_pair(i + 1)
        want = O.hpaged_attention(q, pr.pool, pr.desc, pr.table, lens, H, cur_kv=new_kv)
        O.hpaged_append(pr.pool, pr.desc, pr.table, new_kv, lens - 1, od)
        out = out_tensor(B, Hq, D, ol.OL_F32)
        ol.ol_hpaged_decode_step(pr.kv, pr.pool_d, to_dev(q), Hq, to_dev(new_kv), gd, lens, to_dev(lens), 0.0, -1,
                                 out, ol.OL_F32, ws, n)
        torch.cuda.synchronize()
        check_out(out_as_f64(out), want, ol.OL_F32)
        pr.check_state()
        lens = lens + 1
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK


@pytest.mark.parametrize("shape", [(2, 2, 16, 128), (2, 3, 8, 64), (1, 1, 64, 256)], ids=["s16d128", "s8d64h3",
                                                                                           "s64d256"])
def test_quantize_selected_pages_matches_oracle(shape):
    B, H, S, D = shape
    M = 4
    pr = Pair(B, H, S, D, M, B * M + 2, seed=404 + S)
    lens = np.array([M * S - 1 - 5 * b for b in range(B)], np.int32)
    pr.fill(lens, lambda b, j: 2 * j + b)
    pr.check_state()
    for k, to in enumerate([(2, 7), (4, 0), (3, 1)]):        # wider and narrower targets, K and V apart
        sel = pr.table.reshape(-1)[k::2][: 3].astype(np.int32)
        valid = np.array([(S - 1 - 3 * i) % (S + 1) for i in range(len(sel))], np.int32)
        kf, vf = FORMATS[to[0]][0], FORMATS[to[1]][1]
        od, gd = O.page_desc(k=kf, v=vf), ol.page_format(k=kf, v=vf)
        O.hpaged_quantize(pr.pool, pr.desc, H, D, sel, valid, od)
        ol.ol_hpaged_quantize(pr.kv, pr.pool_d, sel, to_dev(sel), valid, to_dev(valid), gd)
        pr.check_state()
    # attention reads the converted pages
    Hq = 2 * H
    q = bf16_from_f32(pr.rng.standard_normal((B, Hq, D)).astype(np.float32))
    ws, n = workspace(B, Hq, H, D)
    out = out_tensor(B, Hq, D, ol.OL_F32)
    ol.ol_hpaged_decode_attention(pr.kv, to_dev(q), Hq, lens, to_dev(lens), None, 0.0, -1, out, ol.OL_F32, ws, n)
    torch.cuda.synchronize()
    check_out(out_as_f64(out), O.hpaged_attention(q, pr.pool, pr.desc, pr.table, lens, H), ol.OL_F32)


def test_empty_calls_write_nothing():
    pr = Pair(2, 2, 16, 128, 4, 8, seed=505)
    od, gd = fmt_pair(1)
    z = np.zeros(2, np.int32)
    ol.ol_hpaged_append(pr.kv, pr.pool_d, to_dev(pr.values(1)), 0, z, to_dev(z), gd)
    e = np.zeros(0, np.int32)
    ol.ol_hpaged_quantize(pr.kv, pr.pool_d, e, to_dev(np.zeros(4, np.int32)), e, to_dev(np.zeros(4, np.int32)), gd)
    pr.check_state()
    empty = ol.hpaged_kv(pr.pool_d, pr.fmt_d, pr.mirror, pr.bt_d, np.zeros((0, 4), np.int32), kv_heads=2,
                         page_size=16, head_dim=128)
    ws, n = workspace(1, 4, 2, 128)
    out = torch.zeros(16, device="cuda:0")
    ol.ol_hpaged_decode_step(empty, pr.pool_d, to_dev(np.zeros(16, np.uint16)), 4, to_dev(np.zeros(16, np.uint16)), gd,
                             e, to_dev(np.zeros(4, np.int32)), 0.0, -1, out, ol.OL_F32, ws, n)
    pr.check_state()


LONG = [  # B, H, S, Hq, lens: several tiles per warp and several splits per (row, kv head)
    (2, 2, 32, 16, [2500, 1700]),
    (3, 1, 16, 1, [4096, 33, 1]),
    (1, 4, 64, 20, [3001]),
]


@pytest.mark.parametrize("shape", LONG, ids=[f"b{s[0]}h{s[1]}s{s[2]}g{s[3] // s[1]}" for s in LONG])
def test_long_rows_with_every_format_match_oracle(shape):
    B, H, S, Hq, lens = shape
    D = 128
    lens = np.array(lens, np.int32)
    M = int(-(-lens.max() // S)) + 1
    pr = Pair(B, H, S, D, M, B * M, seed=606 + S)
    pr.fill(lens, lambda b, j: (5 * j + 3 * b) % 7 + (j % 3 == 0))
    q = bf16_from_f32(pr.rng.standard_normal((B, Hq, D)).astype(np.float32))
    ws, n = workspace(B, Hq, H, D)
    for window in (-1, 700):
        out = out_tensor(B, Hq, D, ol.OL_BF16)
        ol.ol_hpaged_decode_attention(pr.kv, to_dev(q), Hq, lens, to_dev(lens), None, 0.0, window, out, ol.OL_BF16,
                                      ws, n)
        torch.cuda.synchronize()
        check_out(out_as_f64(out), O.hpaged_attention(q, pr.pool, pr.desc, pr.table, lens, H, window=window),
                  ol.OL_BF16)
    # a fused step on top: the new token starts or continues its page
    new_kv = pr.values(1)
    od, gd = fmt_pair(4)
    want = O.hpaged_attention(q, pr.pool, pr.desc, pr.table, lens + 1, H, cur_kv=new_kv)
    O.hpaged_append(pr.pool, pr.desc, pr.table, new_kv, lens, od)
    out = out_tensor(B, Hq, D, ol.OL_F32)
    ol.ol_hpaged_decode_step(pr.kv, pr.pool_d, to_dev(q), Hq, to_dev(new_kv), gd, lens + 1, to_dev(lens + 1), 0.0, -1,
                             out, ol.OL_F32, ws, n)
    torch.cuda.synchronize()
    check_out(out_as_f64(out), want, ol.OL_F32)
    pr.check_state()
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK


CHUNKS = [  # B, H, S, D, Hq, lens (before the chunk is counted in), chunk length
    # head_dim 128, pages of 16: tensor-core kernel, 8 / group query tokens per CTA
    (3, 2, 16, 128, 8, [16, 21, 40], 4),
    (2, 1, 4, 64, 4, [3, 9], 5),
    (1, 2, 16, 128, 14, [100], 16),
    (2, 2, 16, 128, 16, [300, 777], 3),
    (2, 4, 32, 128, 8, [64, 500], 8),
    (1, 3, 16, 128, 3, [250], 6),
]


@pytest.mark.parametrize("window", [-1, 0, 7])
@pytest.mark.parametrize("shape", CHUNKS, ids=[f"b{s[0]}s{s[2]}d{s[3]}t{s[6]}" for s in CHUNKS])
def test_chunk_step_matches_oracle(shape, window):
    B, H, S, D, Hq, hist, T = shape
    hist = np.array(hist, np.int32)
    M = int(-(-(hist.max() + T) // S)) + 1
    pr = Pair(B, H, S, D, M, B * M + 1, seed=707 + D + T)
    pr.fill(hist, lambda b, j: 2 * j + b + 1)
    lens = hist + T
    q = bf16_from_f32(pr.rng.standard_normal((B, Hq, T, D)).astype(np.float32))
    new_kv = pr.values(T)
    od, gd = fmt_pair(5)
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
