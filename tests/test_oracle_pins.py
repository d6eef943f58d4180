"""Pins for the CPU oracle: each test ties one oracle function to something
other than the oracle itself — a figure printed on the pages (tests/golden/),
a closed form, an invariant, or an exhaustive check against an independent
formulation — so that a dropped term, a wrong sign or index, or a transposed
operand in the oracle fails here.
"""
import math
import os

import numpy as np
import pytest

import oracle as O
from workloads import bf16_from_f32, bf16_to_f32, fixture_signed_ramp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


def _f32_cache(B, H, C, D, fill=np.nan):
    return np.full((2, B, H, C, D), fill, dtype=np.float32)


# ------------------------------------------------------------------ attention


def test_single_visible_token_returns_its_value():
    # softmax over one token has weight exactly 1, so y = v_0 exactly
    rng = np.random.default_rng(1)
    cache = _f32_cache(1, 1, 8, 8)
    cache[:, 0, 0, 0] = rng.uniform(-1, 1, size=(2, 8))
    q = rng.uniform(-1, 1, size=(1, 3, 8)).astype(np.float32)
    y = O.decode_attention(q, cache, [1])
    for h in range(3):
        np.testing.assert_array_equal(y[0, h], cache[1, 0, 0, 0].astype(np.float64))


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    n, D = 7, 16
    cache = _f32_cache(1, 1, 16, D)
    cache[0, 0, 0, :n] = rng.uniform(-1, 1, size=D)          # the same key at every position
    cache[1, 0, 0, :n] = rng.uniform(-1, 1, size=(n, D))
    q = rng.uniform(-3, 3, size=(1, 2, D)).astype(np.float32)
    y = O.decode_attention(q, cache, [n])
    want = cache[1, 0, 0, :n].astype(np.float64).mean(axis=0)
    for h in range(2):
        np.testing.assert_allclose(y[0, h], want, rtol=0, atol=1e-12)


def test_two_token_logistic_pins_scale_and_sign():
    # D = 4, default scale 1/sqrt(4) = 1/2. q = (a,0,0,0), k0 = (1,0,0,0), k1 = 0:
    # s0 = a/2, s1 = 0, so w0 = 1 / (1 + exp(-a/2)); a = 2 ln 3 gives w0 = 3/4.
    a = np.float32(2.0 * math.log(3.0))
    cache = _f32_cache(1, 1, 4, 4)
    cache[0, 0, 0, 0] = [1, 0, 0, 0]
    cache[0, 0, 0, 1] = [0, 0, 0, 0]
    cache[1, 0, 0, 0] = [1, 0, 0, 0]
    cache[1, 0, 0, 1] = [0, 1, 0, 0]
    q = np.array([[[a, 0, 0, 0]]], dtype=np.float32)
    y = O.decode_attention(q, cache, [2])
    w0 = 1.0 / (1.0 + math.exp(-float(a) / 2.0))
    np.testing.assert_allclose(y[0, 0], [w0, 1 - w0, 0, 0], rtol=0, atol=1e-14)
    assert abs(w0 - 0.75) < 1e-6
    # an explicit scale overrides the default: scale 1 gives w0 = 1/(1+exp(-a)) = 9/10
    y1 = O.decode_attention(q, cache, [2], scale=1.0)
    np.testing.assert_allclose(y1[0, 0, 0], 0.9, atol=1e-6)


def test_gqa_contiguous_head_groups():
    # Hq = 6, Hkv = 3 (G = 2): query head h reads kv head h // 2. With V constant
    # per kv head (value g + 1), y[h] = h // 2 + 1 for any q and K.
    rng = np.random.default_rng(3)
    cache = _f32_cache(1, 3, 8, 4)
    cache[0, 0, :, :5] = rng.uniform(-1, 1, size=(3, 5, 4))
    for g in range(3):
        cache[1, 0, g, :5] = g + 1.0
    q = rng.uniform(-1, 1, size=(1, 6, 4)).astype(np.float32)
    y = O.decode_attention(q, cache, [5])
    for h in range(6):
        np.testing.assert_allclose(y[0, h], np.full(4, h // 2 + 1.0), atol=1e-12)


def test_weights_sum_to_one():
    # V = 1 everywhere gives y = sum_t w_t = 1
    rng = np.random.default_rng(4)
    cache = _f32_cache(2, 2, 64, 8)
    cache[0] = rng.uniform(-2, 2, size=cache[0].shape)
    cache[1] = 1.0
    q = rng.uniform(-2, 2, size=(2, 4, 8)).astype(np.float32)
    y = O.decode_attention(q, cache, [64, 33])
    np.testing.assert_allclose(y, 1.0, atol=1e-12)


def test_large_scores_do_not_overflow():
    # scores of order 1e4 would overflow exp() without the max subtraction
    cache = _f32_cache(1, 1, 4, 2)
    cache[0, 0, 0, :3] = [[100, 0], [101, 0], [99, 0]]
    cache[1, 0, 0, :3] = [[1, 0], [2, 0], [3, 0]]
    q = np.array([[[200, 0]]], dtype=np.float32)
    y = O.decode_attention(q, cache, [3])
    assert np.all(np.isfinite(y))
    np.testing.assert_allclose(y[0, 0], [2, 0], atol=1e-12)


def test_causal_prefix_ignores_spare_capacity():
    rng = np.random.default_rng(5)
    C, D = 32, 8
    cache = _f32_cache(2, 2, C, D)
    lens = np.array([9, 20], np.int32)
    for b in range(2):
        cache[:, b, :, : lens[b]] = rng.uniform(-1, 1, size=(2, 2, lens[b], D))
    q = rng.uniform(-1, 1, size=(2, 4, D)).astype(np.float32)
    y = O.decode_attention(q, cache, lens)
    assert np.all(np.isfinite(y))                          # NaN poison beyond lens never read
    cache2 = cache.copy()
    cache2[:, 0, :, 9:] = 7.0                              # rewrite the spare capacity
    np.testing.assert_array_equal(O.decode_attention(q, cache2, lens), y)
    cache3 = cache.copy()
    cache3[1, 0, 0, 8] += 0.5                              # the last visible token does count
    assert not np.array_equal(O.decode_attention(q, cache3, lens)[0, :2], y[0, :2])


def test_token_order_does_not_matter():
    rng = np.random.default_rng(6)
    n, D = 11, 8
    cache = _f32_cache(1, 1, n, D)
    cache[:, 0, 0] = rng.uniform(-1, 1, size=(2, n, D))
    q = rng.uniform(-1, 1, size=(1, 2, D)).astype(np.float32)
    perm = rng.permutation(n)
    cache_p = cache.copy()
    cache_p[:, 0, 0] = cache[:, 0, 0, perm]
    np.testing.assert_allclose(O.decode_attention(q, cache_p, [n]), O.decode_attention(q, cache, [n]),
                               atol=1e-14)


def test_window_zero_and_one():
    rng = np.random.default_rng(7)
    n, D = 10, 8
    cache = _f32_cache(1, 1, 16, D)
    cache[:, 0, 0, :n] = rng.uniform(-1, 1, size=(2, n, D))
    q = rng.uniform(-1, 1, size=(1, 1, D)).astype(np.float32)
    y0 = O.decode_attention(q, cache, [n], window=0)       # only the current token
    np.testing.assert_array_equal(y0[0, 0], cache[1, 0, 0, n - 1].astype(np.float64))
    # window 1 over n tokens equals unbounded attention over the last two tokens alone
    y1 = O.decode_attention(q, cache, [n], window=1)
    tail = _f32_cache(1, 1, 2, D)
    tail[:, 0, 0] = cache[:, 0, 0, n - 2 : n]
    np.testing.assert_allclose(y1, O.decode_attention(q, tail, [2]), atol=1e-15)
    cache_poison = cache.copy()
    cache_poison[:, 0, 0, : n - 2] = np.nan                # tokens left of the window are never read
    np.testing.assert_array_equal(O.decode_attention(q, cache_poison, [n], window=1), y1)


def test_window_visibility_matches_windowed_fixture_bytes():
    g = {k: v for k, *v in _golden_lines("page_counts.txt")}
    retained = int(g["windowed_retained"][0])
    appended = int(g["windowed_appended"][0])
    w = int(g["windowed_window"][0])
    dk, dv = int(g["windowed_dk"][0]), int(g["windowed_dv"][0])
    decoded = 0
    for i in range(appended):                 # query i sits at position retained + i
        lo, hi = O.visible_range(retained + i + 1, w)
        decoded += (hi - lo) * (dk + dv) * 4  # FLOAT bytes
    assert decoded == int(g["windowed_decoded_bytes"][0])
    assert O.visible_range(5, -1) == (0, 5)
    assert O.visible_range(0, -1) == (0, 0)
    assert O.visible_range(3, 10) == (0, 3)


def test_empty_row_gives_zero():
    cache = _f32_cache(1, 1, 4, 4)
    q = np.ones((1, 1, 4), np.float32)
    np.testing.assert_array_equal(O.decode_attention(q, cache, [0]), 0.0)


def test_bf16_inputs_widen_exactly():
    # bf16 and its exact float32 widening give the same result
    rng = np.random.default_rng(8)
    kv = bf16_from_f32(rng.standard_normal((2, 1, 2, 16, 8)).astype(np.float32))
    q = bf16_from_f32(rng.standard_normal((1, 4, 8)).astype(np.float32))
    y16 = O.decode_attention(q, kv, [13])
    y32 = O.decode_attention(bf16_to_f32(q), bf16_to_f32(kv), [13])
    np.testing.assert_array_equal(y16, y32)


def test_paged_equals_contiguous():
    rng = np.random.default_rng(9)
    B, Hkv, Hq, S, D, M, P = 3, 2, 6, 4, 8, 5, 32
    lens = np.array([1, 13, 20], np.int32)
    contiguous = _f32_cache(B, Hkv, M * S, D)
    for b in range(B):
        contiguous[:, b, :, : lens[b]] = rng.uniform(-1, 1, size=(2, Hkv, lens[b], D))
    table = rng.permutation(P)[: B * M].reshape(B, M).astype(np.int32)
    pool = np.full((2, P, Hkv, S, D), np.nan, np.float32)
    # place logical token t of row b by hand: page table[b, t // S], slot t % S
    for b in range(B):
        for t in range(lens[b]):
            pool[:, table[b, t // S], :, t % S] = contiguous[:, b, :, t]
    q = rng.uniform(-1, 1, size=(B, Hq, D)).astype(np.float32)
    for w in (-1, 0, 5):
        np.testing.assert_array_equal(O.paged_attention(q, pool, table, lens, window=w),
                                      O.decode_attention(q, contiguous, lens, window=w))


def test_paged_attention_rejects_out_of_range_page():
    pool = np.zeros((2, 4, 1, 4, 4), np.float32)
    table = np.array([[0, 9]], np.int32)
    q = np.zeros((1, 1, 4), np.float32)
    with pytest.raises(O.OracleError):
        O.paged_attention(q, pool, table, [6])
    O.paged_attention(q, pool, table, [4])     # page 9 is never reached


# -------------------------------------------------------------------- appends


def test_cache_update_writes_only_target_rows():
    rng = np.random.default_rng(10)
    B, H, C, D, L = 3, 2, 12, 4, 2
    cache = rng.uniform(-1, 1, size=(2, B, H, C, D)).astype(np.float32)
    before = cache.copy()
    values = rng.uniform(-1, 1, size=(2, B, H, L, D)).astype(np.float32)
    pos = np.array([0, 5, 10], np.int32)
    O.cache_update(cache, values, pos)
    for b in range(B):
        for t in range(C):
            if pos[b] <= t < pos[b] + L:
                np.testing.assert_array_equal(cache[:, b, :, t], values[:, b, :, t - pos[b]])
            else:
                np.testing.assert_array_equal(cache[:, b, :, t], before[:, b, :, t])


def test_cache_update_rejects_overflow_without_writing():
    cache = np.zeros((2, 2, 1, 8, 4), np.float32)
    values = np.ones((2, 2, 1, 2, 4), np.float32)
    with pytest.raises(O.OracleError):
        O.cache_update(cache, values, [0, 7])            # row 1: 7 + 2 > 8
    np.testing.assert_array_equal(cache, 0.0)            # row 0 untouched as well
    with pytest.raises(O.OracleError):
        O.cache_update(cache, values, [-1, 0])
    O.cache_update(cache, values, [0, 6])                # 6 + 2 == capacity is legal


def test_append_bytes_match_pages_table():
    g = {k: v for k, *v in _golden_lines("page_counts.txt")}
    # FLOAT K/V with Dk = Dv = 2: 4 * (Dk + Dv) = 16 bytes per token
    C, D = 8, 2
    cache = np.zeros((2, 1, 1, C, D), np.float32)
    rng = np.random.default_rng(11)
    retained = []
    for t in range(4):
        before = cache.copy()
        values = rng.uniform(0.5, 1.0, size=(2, 1, 1, 1, D)).astype(np.float32)
        O.cache_update(cache, values, [t])
        changed = np.count_nonzero(before.view(np.uint8) != cache.view(np.uint8))
        assert changed == int(g["append_bytes_per_token_f32_dk2_dv2"][0])
        retained.append((t + 1) * 2 * D * 4)            # valid tokens x bytes per token
    assert retained == [int(x) for x in g["retained_bytes_after_tokens"]]


def test_paged_update_places_page_and_slot():
    rng = np.random.default_rng(12)
    B, H, S, D, M, P, L = 2, 2, 4, 3, 4, 16, 3
    table = rng.permutation(P)[: B * M].reshape(B, M).astype(np.int32)
    pool = np.zeros((2, P, H, S, D), np.float32)
    values = rng.uniform(-1, 1, size=(2, B, H, L, D)).astype(np.float32)
    pos = np.array([2, 9], np.int32)
    O.paged_update(pool, table, values, pos)
    for b in range(B):
        for j in range(L):
            t = pos[b] + j
            np.testing.assert_array_equal(pool[:, table[b, t // S], :, t % S], values[:, b, :, j])
    assert np.count_nonzero(pool) == values.size         # nothing else written


def test_paged_update_rejects_bad_page_without_writing():
    pool = np.zeros((2, 4, 1, 4, 2), np.float32)
    table = np.array([[1, -1], [2, 3]], np.int32)
    values = np.ones((2, 2, 1, 1, 2), np.float32)
    with pytest.raises(O.OracleError):
        O.paged_update(pool, table, values, [4, 0])      # row 0 reaches page -1
    np.testing.assert_array_equal(pool, 0.0)
    with pytest.raises(O.OracleError):
        O.paged_update(pool, table, values, [0, 8])      # beyond M * S
    np.testing.assert_array_equal(pool, 0.0)


# ----------------------------------------------------------------------- INT4


def test_pack_golden():
    for kind, *rest in _golden_lines("packing.txt"):
        if kind == "pack":
            arrow = rest.index("->")
            codes = [int(x) for x in rest[:arrow]]
            hexes = rest[arrow + 1:]
            packed = O.pack_u4(codes)
            assert [f"{b:02x}" for b in packed] == hexes
            np.testing.assert_array_equal(O.unpack_u4(packed, len(codes)), codes)
        elif kind == "size":
            n, nbytes = int(rest[0]), int(rest[1])
            assert O.pack_u4(np.zeros(n, np.uint8)).size == nbytes


def test_int4_row_sizes():
    # 128 dims: 64 code bytes (two per byte), 4 fp16 scales, two zero points per byte
    assert O.int4_row_bytes(128) == (64, 4, 2)
    assert O.int4_row_bytes(32) == (16, 1, 1)


def test_fixed_parameters_golden_ties():
    for x, code in _golden_lines("int4_fixed_ties.txt"):
        row = np.zeros(32, np.float32)
        row[0] = float(x)
        codes, scales, zps = O.int4_quantize_row(bf16_from_f32(row), mode=O.Q_FIXED)
        assert O.unpack_u4(codes, 32)[0] == int(code), x
        assert O.fp16_to_float(scales[0]) == 0.25 and (zps[0] & 0xF) == 8


@pytest.mark.parametrize("zp", [8, 7, 0, 15])
def test_fixed_parameters_exhaustive_over_bf16(zp):
    # every finite bf16 value: code = clamp(round_half_even(x / 0.25) + zp, 0, 15), with x / 0.25 = 4x
    # computed exactly in Python and rounded by Python's round() (ties to even). An odd zero point
    # separates "round, then add zp" (the QuantizeLinear order) from "add zp, then round" at ties.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bf16_to_f32(bits)
    finite = np.isfinite(x)
    bits = np.where(finite, bits, 0).astype(np.uint16)
    x = bf16_to_f32(bits).astype(np.float64)
    got = np.empty(65536, np.uint8)
    for i in range(0, 65536, 32):
        codes, _, zps = O.int4_quantize_row(bits[i : i + 32], mode=O.Q_FIXED, fixed_zp=zp)
        got[i : i + 32] = O.unpack_u4(codes, 32)
        assert zps[0] & 0xF == zp
    want = np.array([min(max(round(v * 4.0) + zp, 0), 15) for v in x], dtype=np.uint8)
    np.testing.assert_array_equal(got, want)


def _dynamic_blocks(seed, nblocks, scale=1.0):
    rng = np.random.default_rng(seed)
    return bf16_from_f32((rng.standard_normal((nblocks, 32)) * scale).astype(np.float32))


def test_dynamic_reconstruction_within_half_scale():
    blocks = _dynamic_blocks(13, 400)
    for row in blocks:
        codes, scales, zps = O.int4_quantize_row(row)
        xhat = O.int4_dequantize_row(codes, scales, zps)
        x = bf16_to_f32(row).astype(np.float64)
        s = O.fp16_to_float(scales[0])
        c = O.unpack_u4(codes, 32)
        inner = (c > 0) & (c < 15)                     # not saturated
        assert np.all(np.abs(xhat - x)[inner] <= s * (0.5 + 1e-6))


def test_dynamic_minimum_maps_to_code_zero_and_maximum_near_top():
    blocks = _dynamic_blocks(14, 400)
    for row in blocks:
        x = bf16_to_f32(row)
        codes, scales, zps = O.int4_quantize_row(row)
        c = O.unpack_u4(codes, 32)
        if x.min() < 0:
            assert c[np.argmin(x)] == 0
        if x.max() > 0:
            assert c[np.argmax(x)] >= 14
        assert np.all(c <= 15)


def test_dynamic_scale_is_fp16_rounding_of_range():
    # the stored scale is the fp16 rounding (numpy's float16 cast, an independent
    # implementation) of the float32 (hi - lo) / 15 with lo, hi including zero
    blocks = _dynamic_blocks(15, 200, scale=3.0)
    for row in blocks:
        x = bf16_to_f32(row)
        lo, hi = np.float32(min(0.0, x.min())), np.float32(max(0.0, x.max()))
        want = np.array([(hi - lo) / np.float32(15.0)], np.float32).astype(np.float16).view(np.uint16)[0]
        _, scales, _ = O.int4_quantize_row(row)
        assert scales[0] == want


def test_all_zero_block_uses_unit_scale():
    codes, scales, zps = O.int4_quantize_row(np.zeros(64, np.uint16))
    assert [O.fp16_to_float(s) for s in scales] == [1.0, 1.0]
    assert np.all(codes == 0) and np.all(zps == 0)


def test_zero_points_pack_two_per_byte_low_first():
    # block 0 all negative, block 1 all positive: zp0 = 15, zp1 = 0 -> byte 0x0f
    row = np.concatenate([np.full(32, -1.0), np.full(32, 1.0)]).astype(np.float32)
    _, scales, zps = O.int4_quantize_row(bf16_from_f32(row))
    assert zps[0] == 0x0F


def test_int4_append_places_rows():
    rng = np.random.default_rng(16)
    B, H, C, D = 2, 2, 6, 64
    codes, scales, zps = O.int4_planes(B, H, C, D)
    values = bf16_from_f32(rng.standard_normal((2, B, H, 1, D)).astype(np.float32))
    O.int4_append(codes, scales, zps, values, [3, 5])
    for k in range(2):
        for b, p in enumerate([3, 5]):
            for h in range(H):
                c, s, z = O.int4_quantize_row(values[k, b, h, 0])
                np.testing.assert_array_equal(codes[k, b, h, p], c)
                np.testing.assert_array_equal(scales[k, b, h, p], s)
                np.testing.assert_array_equal(zps[k, b, h, p], z)
    assert np.count_nonzero(codes[:, 0, :, [0, 1, 2, 4, 5]]) == 0
    with pytest.raises(O.OracleError):
        O.int4_append(codes, scales, zps, values, [6, 0])


def _dense_from_int4(codes, scales, zps, lens, D):
    """Reconstructed values as a float32 contiguous cache (exact: (c - zp) * fp16 scale fits fp32)."""
    _, B, H, C, _ = codes.shape
    out = np.full((2, B, H, C, D), np.nan, np.float32)
    for k in range(2):
        for b in range(B):
            for h in range(H):
                for t in range(lens[b]):
                    out[k, b, h, t] = O.int4_dequantize_row(codes[k, b, h, t], scales[k, b, h, t],
                                                            zps[k, b, h, t]).astype(np.float32)
    return out


def test_int4_attention_equals_dense_attention_on_reconstructed_values():
    # page "Persistent input/output feedback": paged consumer vs dense Attention on the
    # reconstructed values, absolute tolerance 1e-5
    rng = np.random.default_rng(17)
    B, Hkv, Hq, C, D = 2, 2, 4, 12, 64
    lens = np.array([12, 5], np.int32)
    codes, scales, zps = O.int4_planes(B, Hkv, C, D)
    for t in range(C):
        vals = bf16_from_f32(rng.standard_normal((2, B, Hkv, 1, D)).astype(np.float32))
        O.int4_append(codes, scales, zps, vals, [t, t])
    q = bf16_from_f32(rng.standard_normal((B, Hq, D)).astype(np.float32))
    dense = _dense_from_int4(codes, scales, zps, lens, D)
    for w in (-1, 2):
        y4 = O.int4_attention(q, codes, scales, zps, lens, window=w)
        yd = O.decode_attention(bf16_to_f32(q), dense, lens, window=w)
        np.testing.assert_allclose(y4, yd, rtol=0, atol=1e-5)


def test_int4_current_token_is_attended_uncompressed():
    rng = np.random.default_rng(18)
    B, Hkv, Hq, C, D = 1, 1, 2, 8, 32
    codes, scales, zps = O.int4_planes(B, Hkv, C, D)
    hist = bf16_from_f32(rng.standard_normal((2, B, Hkv, 4, D)).astype(np.float32))
    O.int4_append(codes, scales, zps, hist, [0])
    cur = bf16_from_f32(rng.standard_normal((2, B, Hkv, 1, D)).astype(np.float32))
    q = bf16_from_f32(rng.standard_normal((B, Hq, D)).astype(np.float32))
    y = O.int4_attention(q, codes, scales, zps, [5], cur_kv=cur)
    dense = _dense_from_int4(codes, scales, zps, [4], D)
    dense[:, 0, 0, 4] = bf16_to_f32(cur[:, 0, 0, 0])
    np.testing.assert_allclose(y, O.decode_attention(bf16_to_f32(q), dense, [5]), atol=1e-12)
    # window 0 with the current token uncompressed returns exactly its V
    y0 = O.int4_attention(q, codes, scales, zps, [5], cur_kv=cur, window=0)
    np.testing.assert_array_equal(y0[0, 0], bf16_to_f32(cur[1, 0, 0, 0]).astype(np.float64))


def test_int4_chunk_of_one_token_is_the_decode_step():
    # a chunk of one token is the decode step with the current token uncompressed
    rng = np.random.default_rng(19)
    B, Hkv, Hq, C, D = 2, 2, 6, 16, 64
    lens = np.array([9, 1], np.int32)
    codes, scales, zps = O.int4_planes(B, Hkv, C, D)
    hist = bf16_from_f32(rng.standard_normal((2, B, Hkv, 8, D)).astype(np.float32))
    O.int4_append(codes, scales, zps, hist, [0, 0])
    cur = bf16_from_f32(rng.standard_normal((2, B, Hkv, 1, D)).astype(np.float32))
    q = bf16_from_f32(rng.standard_normal((B, Hq, D)).astype(np.float32))
    for w in (-1, 0, 3):
        y = O.int4_chunk_attention(q[:, :, None, :], codes, scales, zps, lens, 1, cur, window=w)
        np.testing.assert_array_equal(y[:, :, 0], O.int4_attention(q, codes, scales, zps, lens, cur_kv=cur,
                                                                      window=w))


def test_int4_chunk_reads_history_from_codes_and_the_chunk_uncompressed():
    # chunk values on the fixed-parameter grid ((k - 8) * 0.25) survive quantization
    # exactly, so attending them uncompressed must equal quantizing the chunk first
    # and attending every token from the codes, one query token at a time
    rng = np.random.default_rng(20)
    B, Hkv, Hq, C, D, T = 2, 2, 4, 20, 64, 4
    lens = np.array([12, 4], np.int32)
    mode = dict(mode=O.Q_FIXED, fixed_scale=0.25, fixed_zp=8)
    codes, scales, zps = O.int4_planes(B, Hkv, C, D)
    hist = bf16_from_f32(rng.standard_normal((2, B, Hkv, 8, D)).astype(np.float32))
    O.int4_append(codes, scales, zps, hist, [0, 0], **mode)
    grid = ((rng.integers(0, 16, (2, B, Hkv, T, D)) - 8) * 0.25).astype(np.float32)
    chunk = bf16_from_f32(grid)
    q = bf16_from_f32(rng.standard_normal((B, Hq, T, D)).astype(np.float32))
    for w in (-1, 2):
        y = O.int4_chunk_attention(q, codes, scales, zps, lens, T, chunk, window=w)
        after = [a.copy() for a in (codes, scales, zps)]
        O.int4_append(*after, chunk, lens - T, **mode)
        for i in range(T):
            yi = O.int4_attention(np.ascontiguousarray(q[:, :, i]), *after, lens - T + i + 1, window=w)
            np.testing.assert_allclose(y[:, :, i], yi, rtol=0, atol=1e-12)
    # query token 0 of the chunk does not see the chunk's later tokens
    moved = chunk.copy()
    moved[:, :, :, 1:] = bf16_from_f32(rng.standard_normal((2, B, Hkv, T - 1, D)).astype(np.float32))
    y0 = O.int4_chunk_attention(q, codes, scales, zps, lens, T, chunk)[:, :, 0]
    np.testing.assert_array_equal(O.int4_chunk_attention(q, codes, scales, zps, lens, T, moved)[:, :, 0], y0)


def test_four_step_fixture_tolerance():
    # page "Persistent input/output feedback", tolerance table: Q/K/V components +/-(0.173*step),
    # UINT4 scale 0.25 / zero point 8, four steps; quantized attention within 0.15 of the
    # unquantized dense attention. Sign pattern (-1)^(d+h) (the page does not print one).
    B, Hkv, Hq, C, D = 1, 1, 2, 8, 64
    codes, scales, zps = O.int4_planes(B, Hkv, C, D)
    dense = np.full((2, B, Hkv, C, D), np.nan, np.float32)
    worst = 0.0
    for step in range(1, 5):
        pos = step - 1
        kv = bf16_from_f32(np.stack([fixture_signed_ramp(B, Hkv, 1, D, step),
                                     fixture_signed_ramp(B, Hkv, 1, D, step)]))
        q = bf16_from_f32(fixture_signed_ramp(B, Hq, 1, D, step)[:, :, 0])
        y4 = O.int4_attention(q, codes, scales, zps, [step], cur_kv=kv)
        O.int4_append(codes, scales, zps, kv, [pos], mode=O.Q_FIXED)
        O.cache_update(dense, bf16_to_f32(kv), [pos])
        yd = O.decode_attention(bf16_to_f32(q), dense, [step])
        worst = max(worst, float(np.abs(y4 - yd).max()))
        # history-only reading (current token from the codes) obeys the same bound
        y4h = O.int4_attention(q, codes, scales, zps, [step])
        worst = max(worst, float(np.abs(y4h - yd).max()))
    assert worst <= 0.15
    assert worst > 0.0                                  # quantization did change the values


# ------------------------------------------------------------ chunked steps

def _causal_brute_force(q, k, v, pos, scale, window):
    """Full score matrix with a causal (and left-window) mask, row softmax,
    weighted sum: written independently of the oracle, in float64.
    q [T, D] for one (row, head); k, v [C, D]; pos [T] query positions."""
    s = (q @ k.T) * scale
    t = np.arange(k.shape[0])[None, :]
    lo = pos[:, None] - (window if window >= 0 else 10 ** 9)
    mask = (t <= pos[:, None]) & (t >= lo)
    s = np.where(mask, s, -np.inf)
    w = np.exp(s - s.max(axis=1, keepdims=True))
    w /= w.sum(axis=1, keepdims=True)
    return w @ v


@pytest.mark.parametrize("window", [-1, 0, 3])
def test_chunk_attention_equals_masked_brute_force(window):
    rng = np.random.default_rng(71)
    B, Hq, Hkv, D, C, T = 2, 4, 2, 8, 12, 3
    cache = rng.standard_normal((2, B, Hkv, C, D)).astype(np.float32)
    q = rng.standard_normal((B, Hq, T, D)).astype(np.float32)
    lens = np.array([T, 10], np.int32)              # row 0: the chunk is the whole row
    y = O.chunk_attention(q, cache, lens, T, window=window)
    scale = 1.0 / math.sqrt(D)
    for b in range(B):
        pos = lens[b] - T + np.arange(T)
        for h in range(Hq):
            g = h // (Hq // Hkv)
            want = _causal_brute_force(q[b, h].astype(np.float64), cache[0, b, g].astype(np.float64),
                                       cache[1, b, g].astype(np.float64), pos, scale, window)
            np.testing.assert_allclose(y[b, h], want, rtol=0, atol=1e-12)


def test_chunk_first_query_ignores_later_chunk_tokens():
    # causality inside the chunk: changing the K/V of chunk tokens 1.. leaves
    # query token 0 unchanged, and changes query token 1
    rng = np.random.default_rng(72)
    B, Hq, Hkv, D, C, T = 1, 2, 1, 8, 16, 3
    cache = rng.standard_normal((2, B, Hkv, C, D)).astype(np.float32)
    q = rng.standard_normal((B, Hq, T, D)).astype(np.float32)
    lens = np.array([9], np.int32)
    y0 = O.chunk_attention(q, cache, lens, T)
    cache2 = cache.copy()
    cache2[:, 0, 0, 7:9] += 5.0                      # chunk tokens 1 and 2 (positions 7, 8)
    y1 = O.chunk_attention(q, cache2, lens, T)
    np.testing.assert_array_equal(y0[:, :, 0], y1[:, :, 0])
    assert np.abs(y0[:, :, 1] - y1[:, :, 1]).max() > 1e-3


def test_paged_chunk_equals_contiguous_chunk():
    rng = np.random.default_rng(73)
    B, Hq, Hkv, D, S, M, T = 2, 4, 2, 8, 4, 5, 4
    C = S * M
    cache = rng.standard_normal((2, B, Hkv, C, D)).astype(np.float32)
    q = rng.standard_normal((B, Hq, T, D)).astype(np.float32)
    perm = rng.permutation(B * M).astype(np.int32)
    table = perm.reshape(B, M)
    pool = np.zeros((2, B * M, Hkv, S, D), np.float32)
    for b in range(B):
        for j in range(M):
            pool[:, table[b, j]] = cache[:, b, :, j * S:(j + 1) * S]
    lens = np.array([7, 20], np.int32)
    np.testing.assert_array_equal(O.paged_chunk_attention(q, pool, table, lens, T, window=5),
                                  O.chunk_attention(q, cache, lens, T, window=5))


# --------------------------------------------------- heterogeneous pages

def test_hf_two_bit_codes_by_hand():
    # INT2, scale 1, zero point 0: saturate(round_half_even(x)) to [-2, 1],
    # two's complement in two bits, four codes per byte, least-significant first
    x = bf16_from_f32(np.array([-3, -2, -1, 0, 1, 2, 0.5, 1.5], np.float32))
    row = O.hf_encode_row(x, (O.HF_I2, 1.0, 0))
    # codes -2 -2 -1 0 -> 0b00_11_10_10 ; codes 1 1 0 1 (0.5 -> 0, 1.5 -> 2 -> 1) -> 0b01_00_01_01
    assert row.tolist() == [0x3A, 0x45]
    np.testing.assert_array_equal(O.hf_decode_row(row, 8, (O.HF_I2, 1.0, 0)), [-2, -2, -1, 0, 1, 1, 0, 1])


def test_hf_four_bit_unsigned_packing_by_hand():
    # UINT4, scale 0.25, zero point 8 (the selector example of the pages): x / 0.25 + 8
    x = bf16_from_f32(np.array([0.0, 0.25, -2.0, 1.75, 5.0, -5.0, 0.125, 0.375], np.float32))
    row = O.hf_encode_row(x, (O.HF_U4, 0.25, 8))
    # codes 8, 9, 0, 15, 15 (sat), 0 (sat), 8 (0.5 -> 0), 10 (1.5 -> 2); low nibble first
    assert row.tolist() == [0x98, 0xF0, 0x0F, 0xA8]


@pytest.mark.parametrize("fmt", ["I8", "U8", "I4", "U4", "I2", "U2"])
def test_hf_ties_to_even_and_saturation(fmt):
    f = getattr(O, "HF_" + fmt)
    qmin, qmax = O.HF_RANGE[f]
    zp = (qmin + qmax + 1) // 2 if qmin == 0 else 0
    scale = 0.5
    # x / scale = k + 0.5 rounds to the even neighbour; beyond the range saturates
    ks = np.arange(qmin - zp - 3, qmax - zp + 3)
    x = (ks + 0.5) * scale
    codes = O.hf_decode_row(O.hf_encode_row(bf16_from_f32(x.astype(np.float32)), (f, scale, zp)), len(x),
                            (f, scale, zp)) / scale + zp
    for k, c in zip(ks, codes):
        want = min(max(int(k) + (int(k) % 2), qmin - zp), qmax - zp) + zp   # even of k, k + 1
        assert c == want, (fmt, k, c, want)


@pytest.mark.parametrize("fmt", ["I8", "U8", "I4", "U4", "I2", "U2"])
def test_hf_reconstruction_within_half_scale(fmt):
    # "each affine reconstruction differs from its source by at most half its scale"
    f = getattr(O, "HF_" + fmt)
    qmin, qmax = O.HF_RANGE[f]
    zp, scale = (qmin + qmax + 1) // 2, 0.125
    rng = np.random.default_rng(81)
    x = rng.uniform((qmin - zp) * scale, (qmax - zp) * scale, 64).astype(np.float32)
    xb = bf16_from_f32(x)
    y = O.hf_decode_row(O.hf_encode_row(xb, (f, scale, zp)), 64, (f, scale, zp))
    assert np.abs(y - bf16_to_f32(xb)).max() <= scale / 2 + 1e-9


def test_hf_dense_formats():
    rng = np.random.default_rng(82)
    x = bf16_from_f32(rng.standard_normal(32).astype(np.float32))
    xf = bf16_to_f32(x).astype(np.float64)
    for f in (O.HF_F32, O.HF_BF16):                  # bf16 values are exact in both
        np.testing.assert_array_equal(O.hf_decode_row(O.hf_encode_row(x, (f, 0, 0)), 32, (f, 0, 0)), xf)
    h = O.hf_decode_row(O.hf_encode_row(x, (O.HF_F16, 0, 0)), 32, (O.HF_F16, 0, 0))
    np.testing.assert_array_equal(h, xf.astype(np.float16).astype(np.float64))   # nearest fp16


def _hetero_case(B=2, H=2, S=4, M=4, D=8, seed=83):
    rng = np.random.default_rng(seed)
    P = B * M
    table = rng.permutation(P).astype(np.int32).reshape(B, M)
    pool, desc = O.hpaged_pool(P, H, S, D)
    return rng, P, table, pool, desc


def test_hpaged_all_bf16_equals_paged_oracle():
    rng, P, table, pool, desc = _hetero_case()
    B, H, S, M, D = 2, 2, 4, 4, 8
    lens = np.array([16, 7], np.int32)
    hist = bf16_from_f32(rng.standard_normal((2, B, H, 16, D)).astype(np.float32))
    O.hpaged_append(pool, desc, table, hist, [0, 0], O.page_desc())
    dense = np.zeros((2, P, H, S, D), np.uint16)
    O.paged_update(dense, table, hist, [0, 0])
    q = bf16_from_f32(rng.standard_normal((B, 4, D)).astype(np.float32))
    for window in (-1, 2):
        np.testing.assert_array_equal(O.hpaged_attention(q, pool, desc, table, lens, H, window=window),
                                      O.paged_attention(q, dense, table, lens, window=window))


def test_hpaged_pages_keep_their_formats():
    # a token that starts a page stamps the call's formats on it; later tokens of
    # that page use the page's formats; earlier pages keep theirs
    rng, P, table, pool, desc = _hetero_case()
    D, H = 8, 2
    vals = bf16_from_f32(rng.standard_normal((2, 2, H, 6, D)).astype(np.float32))
    O.hpaged_append(pool, desc, table, vals, [0, 0], O.page_desc(k=(O.HF_I8, 0.01, 0), v=(O.HF_U4, 0.25, 8)))
    more = bf16_from_f32(rng.standard_normal((2, 2, H, 3, D)).astype(np.float32))
    O.hpaged_append(pool, desc, table, more, [6, 6], O.page_desc(k=(O.HF_F32, 1, 0), v=(O.HF_I2, 0.5, 0)))
    for b in range(2):
        assert desc["kf"][table[b, 0]] == O.HF_I8 and desc["vf"][table[b, 1]] == O.HF_U4   # slots 0..3, 4..7
        assert desc["kf"][table[b, 2]] == O.HF_F32 and desc["vf"][table[b, 2]] == O.HF_I2  # started at 8


@pytest.mark.parametrize("fmt,scale,zps,tol", [("I8", 0.01, 0, 0.01), ("U8", 0.01, 128, 0.01),
                                               ("I4", 0.25, 0, 0.15), ("U4", 0.25, 8, 0.15)])
def test_hpaged_four_step_fixture_tolerance(fmt, scale, zps, tol):
    # the pages' tolerance table: Q/K/V components +/-(0.173 * step), four steps,
    # K and V stored in `fmt` with scalar (scale, zero point); the current token
    # attended uncompressed; within `tol` of unquantized dense attention
    B, H, Hq, S, M, D = 1, 1, 2, 4, 2, 64
    f = (getattr(O, "HF_" + fmt), scale, zps)
    table = np.arange(M, dtype=np.int32).reshape(1, M)
    pool, desc = O.hpaged_pool(M, H, S, D)
    dense = np.full((2, B, H, S * M, D), np.nan, np.float32)
    worst = 0.0
    for step in range(1, 5):
        kv = bf16_from_f32(np.stack([fixture_signed_ramp(B, H, 1, D, step), fixture_signed_ramp(B, H, 1, D, step)]))
        q = bf16_from_f32(fixture_signed_ramp(B, Hq, 1, D, step)[:, :, 0])
        yq = O.hpaged_attention(q, pool, desc, table, [step], H, cur_kv=kv)
        O.hpaged_append(pool, desc, table, kv, [step - 1], O.page_desc(k=f, v=f))
        O.cache_update(dense, bf16_to_f32(kv), [step - 1])
        yd = O.decode_attention(bf16_to_f32(q), dense, [step])
        worst = max(worst, float(np.abs(yq - yd).max()),
                    float(np.abs(O.hpaged_attention(q, pool, desc, table, [step], H) - yd).max()))
    assert worst <= tol
    assert worst > 0.0


def test_hpaged_chunk_of_one_token_is_the_decode_step():
    rng, P, table, pool, desc = _hetero_case()
    B, H, S, M, D = 2, 2, 4, 4, 8
    hist = bf16_from_f32(rng.standard_normal((2, B, H, 9, D)).astype(np.float32))
    O.hpaged_append(pool, desc, table, hist[:, :, :, :5], [0, 0], O.page_desc(k=(O.HF_I8, 0.02, 3), v=(O.HF_U4, 0.3, 8)))
    O.hpaged_append(pool, desc, table, hist[:, :, :, 5:], [5, 5], O.page_desc(k=(O.HF_F16, 1, 0), v=(O.HF_I2, 0.9, 0)))
    cur = bf16_from_f32(rng.standard_normal((2, B, H, 1, D)).astype(np.float32))
    q = bf16_from_f32(rng.standard_normal((B, 4, D)).astype(np.float32))
    lens = np.array([10, 6], np.int32)
    for w in (-1, 0, 3):
        y = O.hpaged_chunk_attention(q[:, :, None, :], pool, desc, table, lens, H, 1, cur, window=w)
        np.testing.assert_array_equal(y[:, :, 0], O.hpaged_attention(q, pool, desc, table, lens, H, cur_kv=cur,
                                                                       window=w))


def test_hpaged_chunk_reads_history_by_page_and_the_chunk_uncompressed():
    # a BFLOAT16 page stores bf16 values exactly: appending the chunk in BFLOAT16 and
    # attending every token from the pages equals attending the chunk uncompressed
    rng, P, table, pool, desc = _hetero_case()
    B, H, S, M, D, T = 2, 2, 4, 4, 8, 3
    hist = bf16_from_f32(rng.standard_normal((2, B, H, 8, D)).astype(np.float32))
    O.hpaged_append(pool, desc, table, hist, [0, 0], O.page_desc(k=(O.HF_U4, 0.4, 7), v=(O.HF_I8, 0.03, -2)))
    chunk = bf16_from_f32(rng.standard_normal((2, B, H, T, D)).astype(np.float32))
    q = bf16_from_f32(rng.standard_normal((B, 4, T, D)).astype(np.float32))
    lens = np.array([11, 7], np.int32)  # both chunks start a page (slot 0), which takes BFLOAT16
    for w in (-1, 2):
        y = O.hpaged_chunk_attention(q, pool, desc, table, lens, H, T, chunk, window=w)
        p2, d2 = pool.copy(), desc.copy()
        O.hpaged_append(p2, d2, table, chunk, lens - T, O.page_desc())
        for i in range(T):
            yi = O.hpaged_attention(np.ascontiguousarray(q[:, :, i]), p2, d2, table, lens - T + i + 1, H, window=w)
            np.testing.assert_allclose(y[:, :, i], yi, rtol=0, atol=1e-12)
    moved = chunk.copy()
    moved[:, :, :, 1:] = bf16_from_f32(rng.standard_normal((2, B, H, T - 1, D)).astype(np.float32))
    y0 = O.hpaged_chunk_attention(q, pool, desc, table, lens, H, T, chunk)[:, :, 0]
    np.testing.assert_array_equal(O.hpaged_chunk_attention(q, pool, desc, table, lens, H, T, moved)[:, :, 0], y0)


def test_hpaged_quantize_selected_pages_only():
    rng, P, table, pool, desc = _hetero_case()
    B, H, S, M, D = 2, 2, 4, 4, 8
    hist = bf16_from_f32(rng.standard_normal((2, B, H, 14, D)).astype(np.float32))
    O.hpaged_append(pool, desc, table, hist, [0, 0], O.page_desc(k=(O.HF_F32, 1, 0), v=(O.HF_BF16, 1, 0)))
    before, dbefore = pool.copy(), desc.copy()
    sel = np.array([table[0, 1], table[1, 3]], np.int32)          # a full page and a half-full one
    valid = np.array([4, 2], np.int32)                            # row 1 holds 14 tokens: page 3 has 2
    to = O.page_desc(k=(O.HF_I4, 0.125, 0), v=(O.HF_U2, 0.5, 2))
    O.hpaged_quantize(pool, desc, H, D, sel, valid, to)
    for p in range(P):
        if p not in sel:
            np.testing.assert_array_equal(pool[p], before[p])
            assert desc[p] == dbefore[p]
    assert desc["kf"][sel[0]] == O.HF_I4 and desc["vf"][sel[1]] == O.HF_U2
    # valid rows reconstruct within half a scale of the source; unused rows are the
    # destination's zeros (code = zero point)
    for p, n in zip(sel, valid):
        for h in range(H):
            for s in range(S):
                for plane, (f, sc, zp) in ((0, (O.HF_I4, 0.125, 0)), (1, (O.HF_U2, 0.5, 2))):
                    rb = D * O.HF_BITS[f] // 8
                    off = plane * H * S * D * 4 + (h * S + s) * rb
                    got = O.hf_decode_row(pool[p, off:off + rb], D, (f, sc, zp))
                    if s >= n:
                        np.testing.assert_array_equal(got, np.zeros(D))
                    else:
                        f0 = (O.HF_F32, 1, 0) if plane == 0 else (O.HF_BF16, 1, 0)
                        rb0 = D * O.HF_BITS[f0[0]] // 8
                        off0 = plane * H * S * D * 4 + (h * S + s) * rb0
                        src = O.hf_decode_row(before[p, off0:off0 + rb0], D, f0)
                        lo, hi = (O.HF_RANGE[f][0] - zp) * sc, (O.HF_RANGE[f][1] - zp) * sc
                        expect = np.clip(src, lo, hi)
                        assert np.abs(got - expect).max() <= sc / 2 + 1e-9
    with pytest.raises(O.OracleError):                             # duplicate index
        O.hpaged_quantize(pool, desc, H, D, np.array([1, 1], np.int32), np.array([4, 4], np.int32), to)
