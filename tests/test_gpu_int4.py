"""GPU parity of the INT4 blockwise-affine path against the CPU oracle.

History is quantized by the oracle from seeded bf16 values. The CUDA step
quantizes and appends the new token (codes, fp16 scales and zero points must
be bit-exact with the oracle's) and attends history from the codes plus the
current token uncompressed; outputs within 2e-3 of the oracle.
"""
import numpy as np
import pytest
import torch

import oracle as O
import place_kv_cache_gb300 as ol
from workloads import Workload, bf16_from_f32, make_case
from tests.gpu_util import check_out, max_abs_err, out_as_f64, out_tensor, to_dev, to_host, workspace

pytestmark = pytest.mark.gpu
TOL = 2e-3
MODES = {"dynamic": O.Q_DYNAMIC, "fixed": O.Q_FIXED}


def oracle_planes(case, mode):
    w = case.workload
    planes = O.int4_planes(w.batch, w.kv_heads, w.capacity, w.head_dim)
    for b, h in enumerate(case.history):
        n = h.shape[2]
        if n == 0:
            continue
        sub = O.int4_planes(1, w.kv_heads, w.capacity, w.head_dim)
        O.int4_append(*sub, h[:, None], [0], mode=mode)
        for full, part in zip(planes, sub):
            full[:, b] = part[:, 0]
    return planes


def dev_planes(planes):
    return tuple(to_dev(p) for p in planes)


def host_planes(dplanes):
    return tuple(to_host(p) for p in dplanes)


def desc_of(dplanes, w, mode, access=ol.OL_READ_WRITE):  # noqa: D401
    return ol.int4_kv(*dplanes, head_dim=w.head_dim, quant_mode=mode, access=access)


@pytest.mark.parametrize("mode", list(MODES), ids=list(MODES))
@pytest.mark.parametrize("shape", [
    ("b3_gqa4", 3, 32, 8, 128, 300, [1, 17, 300]),
    ("b2_gqa7", 2, 28, 4, 128, 160, [160, 64]),
    ("b2_gqa5", 2, 10, 2, 128, 150, [150, 20]),
    ("b2_gqa3", 2, 12, 4, 128, 180, [180, 40]),
    ("b2_gqa2", 2, 8, 4, 128, 200, [200, 33]),
    ("b2_gqa1", 2, 4, 4, 128, 130, [130, 5]),
    ("b2_d64", 2, 8, 2, 64, 96, [96, 33]),
    ("b1_d256_gqa1", 1, 2, 2, 256, 64, [50]),
], ids=lambda s: s[0])
def test_int4_step_matches_oracle(shape, mode):
    name, B, Hq, Hkv, D, C, lens = shape
    w = Workload(name, "bf16", B, Hq, Hkv, D, C, "int4", seed=31)
    case = make_case(w, lens=np.array(lens, np.int32))
    qm = MODES[mode]
    planes = oracle_planes(case, qm)
    dplanes = dev_planes(planes)
    ptr0 = dplanes[0].data_ptr()
    ws, n = workspace(B, Hq, Hkv, D)
    out = out_tensor(B, Hq, D, ol.OL_F32)
    ol.ol_decode_step(ol.OL_LAYOUT_INT4, desc_of(dplanes, w, qm), dplanes[0], to_dev(case.q), Hq,
                      to_dev(case.new_kv), case.lens, to_dev(case.lens), 0.0, -1, out, ol.OL_F32, ws, n)
    torch.cuda.synchronize()
    assert dplanes[0].data_ptr() == ptr0
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    O.int4_append(*planes, case.new_kv, case.lens - 1, mode=qm)
    for g, r in zip(host_planes(dplanes), planes):
        np.testing.assert_array_equal(g, r)
    want = O.int4_attention(case.q, *planes, case.lens, cur_kv=case.new_kv)
    assert max_abs_err(out_as_f64(out), want) <= TOL


@pytest.mark.parametrize("window", [-1, 0, 3, 40])
@pytest.mark.parametrize("with_cur", [False, True], ids=["codes_only", "cur_uncompressed"])
def test_int4_attention_read_only(window, with_cur):
    w = Workload("i4a", "bf16", 3, 16, 4, 128, 200, "int4", seed=32)
    case = make_case(w, lens=np.array([200, 1, 57], np.int32), history_len_offset=0)
    planes = oracle_planes(case, O.Q_DYNAMIC)
    dplanes = dev_planes(planes)
    ws, n = workspace(3, 16, 4, 128)
    out = out_tensor(3, 16, 128, ol.OL_BF16)
    cur = case.new_kv if with_cur else None
    ol.ol_int4kv_decode_attention(desc_of(dplanes, w, O.Q_DYNAMIC, access=ol.OL_READ_ONLY), to_dev(case.q), 16,
                                  case.lens, to_dev(case.lens), None if cur is None else to_dev(cur), 0.0, window,
                                  out, ol.OL_BF16, ws, n)
    torch.cuda.synchronize()
    for g, r in zip(host_planes(dplanes), planes):
        np.testing.assert_array_equal(g, r)
    want = O.int4_attention(case.q, *planes, case.lens, cur_kv=cur, window=window)
    check_out(out_as_f64(out), want, ol.OL_BF16)


@pytest.mark.parametrize("mode", list(MODES), ids=list(MODES))
def test_int4_append_codes_bit_exact(mode):
    # wide value ranges, ties and all-zero blocks: every code, scale and zero point bit-exact
    B, H, C, D = 4, 2, 8, 128
    rng = np.random.default_rng(33)
    x = rng.standard_normal((2, B, H, 1, D)).astype(np.float32) * rng.choice([1e-3, 1.0, 30.0], (2, B, H, 1, 1))
    x = x.astype(np.float32)
    x[0, 0, 0, 0, :32] = 0.0                                  # an all-zero block
    x[1, 1, 1, 0, :32] = np.arange(32) * 0.125 - 2.0          # exact ties under scale 0.25
    vals = bf16_from_f32(x)
    qm = MODES[mode]
    planes = O.int4_planes(B, H, C, D)
    dplanes = dev_planes(planes)
    pos = np.array([0, 3, 7, 5], np.int32)
    desc = ol.int4_kv(*dplanes, head_dim=D, quant_mode=qm)
    ol.ol_int4kv_append(desc, dplanes[0], to_dev(vals), pos, to_dev(pos))
    torch.cuda.synchronize()
    O.int4_append(*planes, vals, pos, mode=qm)
    for g, r in zip(host_planes(dplanes), planes):
        np.testing.assert_array_equal(g, r)


def test_int4_chained_steps():
    # eight chained steps carrying the INT4 cache as persistent state
    B, Hq, Hkv, D, C = 2, 8, 2, 128, 96
    w = Workload("chain", "bf16", B, Hq, Hkv, D, C, "int4", seed=34)
    case = make_case(w, lens=np.array([40, 70], np.int32))
    planes = oracle_planes(case, O.Q_DYNAMIC)
    dplanes = dev_planes(planes)
    desc = desc_of(dplanes, w, O.Q_DYNAMIC)
    ws, n = workspace(B, Hq, Hkv, D)
    rng = np.random.default_rng(35)
    lens = case.lens.copy()
    for step in range(8):
        q = bf16_from_f32(rng.standard_normal((B, Hq, D)).astype(np.float32))
        kv = bf16_from_f32(rng.standard_normal((2, B, Hkv, 1, D)).astype(np.float32))
        out = out_tensor(B, Hq, D, ol.OL_F32)
        ol.ol_decode_step(ol.OL_LAYOUT_INT4, desc, dplanes[0], to_dev(q), Hq, to_dev(kv), lens, to_dev(lens), 0.0,
                          -1, out, ol.OL_F32, ws, n)
        torch.cuda.synchronize()
        O.int4_append(*planes, kv, lens - 1)
        want = O.int4_attention(q, *planes, lens, cur_kv=kv)
        assert max_abs_err(out_as_f64(out), want) <= TOL
        lens = lens + 1
    for g, r in zip(host_planes(dplanes), planes):
        np.testing.assert_array_equal(g, r)


def test_int4_history_stable_flag():
    B, Hq, Hkv, D, C = 3, 32, 8, 128, 300
    w = Workload("i4flag", "bf16", B, Hq, Hkv, D, C, "int4", seed=36)
    case = make_case(w, lens=np.array([1, 17, 300], np.int32))
    planes = oracle_planes(case, O.Q_DYNAMIC)
    dplanes = dev_planes(planes)
    ws, n = workspace(B, Hq, Hkv, D)
    out = out_tensor(B, Hq, D, ol.OL_F32)
    desc = desc_of(dplanes, w, O.Q_DYNAMIC, access=ol.OL_READ_WRITE | ol.OL_HISTORY_STABLE)
    ol.ol_decode_step(ol.OL_LAYOUT_INT4, desc, dplanes[0], to_dev(case.q), Hq, to_dev(case.new_kv), case.lens,
                      to_dev(case.lens), 0.0, -1, out, ol.OL_F32, ws, n)
    torch.cuda.synchronize()
    O.int4_append(*planes, case.new_kv, case.lens - 1)
    for g, r in zip(host_planes(dplanes), planes):
        np.testing.assert_array_equal(g, r)
    check_out(out_as_f64(out), O.int4_attention(case.q, *planes, case.lens, cur_kv=case.new_kv), ol.OL_F32)


@pytest.mark.parametrize("shape", [
    # long rows and one short one: each of the ~300 CTAs takes ~70 tiles of the
    # concatenated rows, so ranges cross (row, kv head) boundaries and the
    # short row's units share CTAs (several segments per CTA)
    ("ragged", 6, [16384, 16384, 16000, 700, 16000, 16000], -1),
    ("window", 8, [16384] * 7 + [700], 12000),
], ids=lambda s: s[0])
def test_int4_streamk_matches_oracle(shape):
    name, B, lens, window = shape
    Hq, Hkv, D, C = 16, 4, 128, 16384
    w = Workload("sk_" + name, "bf16", B, Hq, Hkv, D, C, "int4", seed=36)
    case = make_case(w, lens=np.array(lens, np.int32))
    planes = oracle_planes(case, O.Q_DYNAMIC)
    dplanes = dev_planes(planes)
    ws, n = workspace(B, Hq, Hkv, D)
    out = out_tensor(B, Hq, D, ol.OL_F32)
    ol.ol_decode_step(ol.OL_LAYOUT_INT4, desc_of(dplanes, w, O.Q_DYNAMIC), dplanes[0], to_dev(case.q), Hq,
                      to_dev(case.new_kv), case.lens, to_dev(case.lens), 0.0, window, out, ol.OL_F32, ws, n)
    torch.cuda.synchronize()
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    O.int4_append(*planes, case.new_kv, case.lens - 1, mode=O.Q_DYNAMIC)
    for g, r in zip(host_planes(dplanes), planes):
        np.testing.assert_array_equal(g, r)
    want = O.int4_attention(case.q, *planes, case.lens, cur_kv=case.new_kv, window=window)
    assert max_abs_err(out_as_f64(out), want) <= TOL


def scaled_bf16(x, std):
    """bf16 bit patterns of std times the bf16 values x (rounded to nearest even)."""
    f = (x.astype(np.uint32) << 16).view(np.float32) * np.float32(std)
    return bf16_from_f32(f.astype(np.float32))


@pytest.mark.parametrize("heads", [(32, 8), (28, 4)], ids=["gqa4", "gqa7"])
@pytest.mark.parametrize("window", [0, 1, 3, -1])
def test_int4_large_values_short_windows(heads, window):
    # values N(0, 3): with few visible tokens nothing averages the rounding of
    # the weights, so the V side's error shows at its full size (a single fp16
    # P^T times the V scale put it at about 2e-3 here)
    Hq, Hkv = heads
    B, D, C = 4, 128, 512
    w = Workload("i4big", "bf16", B, Hq, Hkv, D, C, "int4", seed=37)
    case = make_case(w, lens=np.array([512, 300, 17, 2], np.int32))
    case.history = [scaled_bf16(h, 3.0) for h in case.history]
    case.new_kv = scaled_bf16(case.new_kv, 3.0)
    planes = oracle_planes(case, O.Q_DYNAMIC)
    dplanes = dev_planes(planes)
    ws, n = workspace(B, Hq, Hkv, D)
    out = out_tensor(B, Hq, D, ol.OL_F32)
    ol.ol_int4kv_decode_attention(desc_of(dplanes, w, O.Q_DYNAMIC, access=ol.OL_READ_ONLY), to_dev(case.q), Hq,
                                  case.lens, to_dev(case.lens), to_dev(case.new_kv), 0.0, window, out, ol.OL_F32,
                                  ws, n)
    torch.cuda.synchronize()
    want = O.int4_attention(case.q, *planes, case.lens, cur_kv=case.new_kv, window=window)
    assert max_abs_err(out_as_f64(out), want) <= TOL
