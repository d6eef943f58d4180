"""Randomised pins for the CPU oracle's attention: closed forms and
invariants checked over drawn shapes (batch, kv heads, query group, head_dim,
capacity, per-row lengths, window), so that an index or stride mistake that
one fixed shape happens to hide (rows and kv heads mixed up, a group mapped
to the wrong kv head, a window off by one at a row boundary) fails here.
Every expected value is a closed form of the definition, an invariant, or
(for chunked steps) a masked-softmax brute force written here, not the
oracle.
"""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle as O  # noqa: E402

SETTINGS = settings(max_examples=60, deadline=None, derandomize=True)


@st.composite
def shapes(draw):
    B = draw(st.integers(1, 3))
    Hkv = draw(st.integers(1, 3))
    G = draw(st.integers(1, 4))
    D = draw(st.sampled_from([4, 8, 16]))
    C = draw(st.integers(1, 24))
    lens = draw(st.lists(st.integers(1, C), min_size=B, max_size=B))
    window = draw(st.sampled_from([-1, 0, 1, 2, 5, 30]))
    seed = draw(st.integers(0, 2**31 - 1))
    return B, Hkv, G, D, C, np.array(lens, np.int32), window, seed


def visible(n, window):
    """Positions the query at p = n - 1 sees: [max(0, p - w), p], or [0, p]."""
    p = n - 1
    lo = 0 if window < 0 else max(0, p - window)
    return lo, p + 1


def nan_cache(B, Hkv, C, D):
    return np.full((2, B, Hkv, C, D), np.nan, np.float32)  # spare capacity poisoned


@SETTINGS
@given(shapes())
def test_identical_keys_in_view_give_the_mean_of_the_visible_values(s):
    B, Hkv, G, D, C, lens, window, seed = s
    rng = np.random.default_rng(seed)
    cache = nan_cache(B, Hkv, C, D)
    want = np.zeros((B, Hkv * G, D))
    for b in range(B):
        lo, hi = visible(lens[b], window)
        for g in range(Hkv):
            cache[0, b, g, :lens[b]] = rng.uniform(-2, 2, size=D)  # one key for the whole row
            cache[1, b, g, :lens[b]] = rng.uniform(-2, 2, size=(lens[b], D))
            want[b, g * G:(g + 1) * G] = cache[1, b, g, lo:hi].astype(np.float64).mean(axis=0)
    q = rng.uniform(-2, 2, size=(B, Hkv * G, D)).astype(np.float32)
    y = O.decode_attention(q, cache, lens, window=window)
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-12)


@SETTINGS
@given(shapes())
def test_a_constant_value_row_is_returned_whatever_the_weights(s):
    # softmax weights sum to one over the visible range, so V constant per
    # (row, kv head) comes back exactly, for any q and K
    B, Hkv, G, D, C, lens, window, seed = s
    rng = np.random.default_rng(seed)
    cache = nan_cache(B, Hkv, C, D)
    want = np.zeros((B, Hkv * G, D))
    for b in range(B):
        for g in range(Hkv):
            v = rng.uniform(-2, 2, size=D).astype(np.float32)
            cache[0, b, g, :lens[b]] = rng.uniform(-3, 3, size=(lens[b], D))
            cache[1, b, g, :lens[b]] = v
            want[b, g * G:(g + 1) * G] = v
    q = rng.uniform(-3, 3, size=(B, Hkv * G, D)).astype(np.float32)
    y = O.decode_attention(q, cache, lens, window=window)
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-12)


@SETTINGS
@given(shapes())
def test_rows_and_kv_heads_are_independent(s):
    # permuting the rows, and the kv heads with their query groups, permutes
    # the outputs the same way
    B, Hkv, G, D, C, lens, window, seed = s
    rng = np.random.default_rng(seed)
    cache = nan_cache(B, Hkv, C, D)
    for b in range(B):
        cache[:, b, :, :lens[b]] = rng.uniform(-2, 2, size=(2, Hkv, lens[b], D))
    q = rng.uniform(-2, 2, size=(B, Hkv * G, D)).astype(np.float32)
    y = O.decode_attention(q, cache, lens, window=window)
    rb = rng.permutation(B)
    rg = rng.permutation(Hkv)
    heads = np.concatenate([np.arange(g * G, (g + 1) * G) for g in rg])
    cache_p = np.ascontiguousarray(cache[:, rb][:, :, rg])
    q_p = np.ascontiguousarray(q[rb][:, heads])
    y_p = O.decode_attention(q_p, cache_p, lens[rb], window=window)
    np.testing.assert_array_equal(y_p, y[rb][:, heads])


@SETTINGS
@given(shapes())
def test_tokens_outside_the_window_do_not_count(s):
    # rewriting every K/V position outside [lo, hi) of every row (spare
    # capacity and positions before the window) leaves y unchanged
    B, Hkv, G, D, C, lens, window, seed = s
    rng = np.random.default_rng(seed)
    cache = rng.uniform(-2, 2, size=(2, B, Hkv, C, D)).astype(np.float32)
    q = rng.uniform(-2, 2, size=(B, Hkv * G, D)).astype(np.float32)
    y = O.decode_attention(q, cache, lens, window=window)
    other = cache.copy()
    for b in range(B):
        lo, hi = visible(lens[b], window)
        other[:, b, :, :lo] = rng.uniform(-50, 50, size=(2, Hkv, lo, D))
        other[:, b, :, hi:] = rng.uniform(-50, 50, size=(2, Hkv, C - hi, D))
    np.testing.assert_array_equal(O.decode_attention(q, other, lens, window=window), y)


@SETTINGS
@given(shapes(), st.integers(1, 4))
def test_paged_layout_equals_contiguous_for_any_page_placement(s, S):
    # the same logical rows scattered over shuffled pages of S slots give the
    # contiguous oracle's result bit for bit
    B, Hkv, G, D, C, lens, window, seed = s
    rng = np.random.default_rng(seed)
    cache = nan_cache(B, Hkv, C, D)
    for b in range(B):
        cache[:, b, :, :lens[b]] = rng.uniform(-2, 2, size=(2, Hkv, lens[b], D))
    q = rng.uniform(-2, 2, size=(B, Hkv * G, D)).astype(np.float32)
    M = (C + S - 1) // S
    P = B * M
    perm = rng.permutation(P)
    table = perm.reshape(B, M).astype(np.int32)
    pool = np.full((2, P, Hkv, S, D), np.nan, np.float32)
    for b in range(B):
        for t in range(lens[b]):
            pool[:, table[b, t // S], :, t % S] = cache[:, b, :, t]
    np.testing.assert_array_equal(O.paged_attention(q, pool, table, lens, window=window),
                                  O.decode_attention(q, cache, lens, window=window))


def _masked_softmax_attention(q, k, v, pos, scale, window):
    """Score matrix with a causal (and left-window) mask, row softmax, weighted
    sum, in float64; written independently of the oracle. q [T, D]; k, v
    [C, D]; pos [T] query positions."""
    s = (q @ k.T) * scale
    t = np.arange(k.shape[0])[None, :]
    lo = pos[:, None] - (window if window >= 0 else 10 ** 9)
    s = np.where((t <= pos[:, None]) & (t >= lo), s, -np.inf)
    w = np.exp(s - s.max(axis=1, keepdims=True))
    return (w / w.sum(axis=1, keepdims=True)) @ v


@SETTINGS
@given(shapes(), st.integers(1, 5), st.floats(0.05, 2.0))
def test_chunk_attention_equals_masked_softmax_over_drawn_shapes(s, T, scale):
    # a chunk of T tokens per row (rows at least T long), any explicit scale
    B, Hkv, G, D, C, lens, window, seed = s
    C = max(C, T)
    lens = np.maximum(np.minimum(lens, C), T).astype(np.int32)
    rng = np.random.default_rng(seed)
    cache = rng.uniform(-2, 2, size=(2, B, Hkv, C, D)).astype(np.float32)
    q = rng.uniform(-2, 2, size=(B, Hkv * G, T, D)).astype(np.float32)
    y = O.chunk_attention(q, cache, lens, T, scale=scale, window=window)
    for b in range(B):
        pos = lens[b] - T + np.arange(T)
        for h in range(Hkv * G):
            g = h // G
            want = _masked_softmax_attention(q[b, h].astype(np.float64), cache[0, b, g].astype(np.float64),
                                             cache[1, b, g].astype(np.float64), pos, scale, window)
            np.testing.assert_allclose(y[b, h], want, rtol=0, atol=1e-12)
