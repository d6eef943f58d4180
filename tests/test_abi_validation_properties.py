"""Randomised CPU tests of the host validation of ol_decode_step (row a1 of
the path: pointer identity, capacity, no buffer over the cache, alignment,
workspace size): drawn shapes and lengths, with at most one violation
planted per request, must give exactly the status the rule names, and every
clean request must pass validation. No GPU is touched: device pointers are
fake aligned addresses, and requests that pass validation stop at the host
fault-injection switch (OL_FAULT_INJECT) before any CUDA call.
"""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import place_kv_cache_gb300 as ol  # noqa: E402

BASE = 0x7E0000000000   # fake device address space
GB = 1 << 30

VIOLATIONS = {
    "none": ol.OL_ERR_INJECTED,
    "len_zero": ol.OL_ERR_CAPACITY,
    "len_over_capacity": ol.OL_ERR_CAPACITY,
    "updated_is_another_pointer": ol.OL_ERR_ALIAS,
    "q_inside_cache": ol.OL_ERR_ALIAS,
    "new_kv_inside_cache": ol.OL_ERR_ALIAS,
    "out_inside_cache": ol.OL_ERR_ALIAS,
    "workspace_inside_cache": ol.OL_ERR_ALIAS,
    "out_over_q": ol.OL_ERR_ALIAS,
    "q_misaligned": ol.OL_ERR_ALIGN,
    "out_misaligned": ol.OL_ERR_ALIGN,
    "workspace_too_small": ol.OL_ERR_WORKSPACE,
    "q_heads_not_a_multiple": ol.OL_ERR_SHAPE,
}


@pytest.fixture(autouse=True)
def _inject(monkeypatch):
    monkeypatch.setenv("OL_FAULT_INJECT", "after_validate")
    yield


@st.composite
def requests(draw):
    B = draw(st.integers(1, 6))
    Hkv = draw(st.integers(1, 4))
    G = draw(st.integers(1, 8))
    D = draw(st.sampled_from([64, 128]))
    C = draw(st.integers(16, 4096))
    lens = draw(st.lists(st.integers(1, C), min_size=B, max_size=B))
    violation = draw(st.sampled_from(sorted(VIOLATIONS)))
    row = draw(st.integers(0, B - 1))
    offset = draw(st.integers(0, 1 << 20))       # where inside the cache a stray buffer starts
    return B, Hkv, G, D, C, lens, violation, row, offset


@settings(max_examples=300, deadline=None, derandomize=True)
@given(requests())
def test_each_rule_gives_its_status(r):
    B, Hkv, G, D, C, lens, violation, row, offset = r
    cache_bytes = 2 * B * Hkv * C * D * 2
    cache = BASE
    q, new_kv, out, lens_dev, ws = (BASE + k * GB for k in (1, 2, 3, 4, 5))
    ws_bytes = ol.ol_workspace_size(B, Hkv * G, Hkv, D)
    q_heads = Hkv * G
    updated = cache
    inside = cache + (offset % cache_bytes) // 16 * 16    # an aligned address inside the cache
    lens = list(lens)
    if violation == "len_zero":
        lens[row] = 0
    elif violation == "len_over_capacity":
        lens[row] = C + 1
    elif violation == "updated_is_another_pointer":
        updated = cache + 16 * (1 + offset % 64)
    elif violation == "q_inside_cache":
        q = inside
    elif violation == "new_kv_inside_cache":
        new_kv = inside
    elif violation == "out_inside_cache":
        out = inside
    elif violation == "workspace_inside_cache":
        ws = inside
    elif violation == "out_over_q":
        out = q + 16 * (offset % 8)
    elif violation == "q_misaligned":
        q += 8
    elif violation == "out_misaligned":
        out += 4
    elif violation == "workspace_too_small":
        ws_bytes -= 1 + offset % 64
    elif violation == "q_heads_not_a_multiple":
        q_heads = Hkv * G + 1 if Hkv > 1 else 0
    desc = ol.kv_cache(cache, dims=(B, Hkv, C, D), dtype=ol.OL_BF16)
    try:
        ol.ol_decode_step(ol.OL_LAYOUT_CONTIGUOUS, desc, updated, q, q_heads, new_kv, np.array(lens, np.int32),
                          lens_dev, 0.0, -1, out, ol.OL_BF16, ws, ws_bytes, stream=0)
        status = ol.OL_OK
    except ol.OlError as e:
        status = e.status
    assert status == VIOLATIONS[violation], (violation, status)


@st.composite
def paged_requests(draw):
    B = draw(st.integers(1, 4))
    Hkv = draw(st.integers(1, 3))
    G = draw(st.integers(1, 4))
    S = draw(st.sampled_from([16, 32]))
    M = draw(st.integers(1, 8))
    P = B * M + draw(st.integers(0, 16))
    lens = draw(st.lists(st.integers(1, M * S), min_size=B, max_size=B))
    case = draw(st.sampled_from(["none", "page_out_of_pool", "page_out_of_pool_not_reached", "append_page_shared",
                                 "history_page_shared", "over_capacity", "updated_is_another_pointer"]))
    seed = draw(st.integers(0, 2**31 - 1))
    return B, Hkv, G, S, M, P, lens, case, seed


@settings(max_examples=300, deadline=None, derandomize=True)
@given(paged_requests())
def test_paged_page_rules_give_their_status(r):
    # a fused step appends at lens - 1 and reads [0, lens - 1): every page a
    # row reaches must lie in the pool, and no row may append into a page
    # another row also reaches; pages beyond a row's length are never looked at
    # and rows may share pages they only read
    B, Hkv, G, S, M, P, lens, case, seed = r
    rng = np.random.default_rng(seed)
    D = 128
    table = rng.permutation(P)[:B * M].reshape(B, M).astype(np.int32)   # distinct pages
    lens = list(lens)
    reached = [(n - 1) // S for n in lens]                               # last page index each row reaches
    pool, bt = BASE, BASE + 6 * GB
    updated = pool
    want = ol.OL_ERR_INJECTED
    b = int(rng.integers(B))
    if case == "page_out_of_pool":
        table[b, int(rng.integers(reached[b] + 1))] = P if rng.integers(2) else -1
        want = ol.OL_ERR_PAGE
    elif case == "page_out_of_pool_not_reached" and reached[b] + 1 < M:
        table[b, int(rng.integers(reached[b] + 1, M))] = P
    elif case == "append_page_shared" and B > 1:
        other = (b + 1 + int(rng.integers(B - 1))) % B
        table[other, int(rng.integers(reached[other] + 1))] = table[b, reached[b]]
        want = ol.OL_ERR_PAGE
    elif case == "history_page_shared" and B > 1:
        other = (b + 1 + int(rng.integers(B - 1))) % B
        if reached[b] >= 1 and reached[other] >= 1:                      # neither row appends into it
            table[other, int(rng.integers(reached[other]))] = table[b, int(rng.integers(reached[b]))]
    elif case == "over_capacity":
        lens[b] = M * S + 1
        want = ol.OL_ERR_CAPACITY
    elif case == "updated_is_another_pointer":
        updated = pool + 16
        want = ol.OL_ERR_ALIAS
    desc = ol.paged_kv(pool, bt, table, dims=(P, Hkv, S, D), dtype=ol.OL_BF16)
    q, new_kv, out, lens_dev, ws = (BASE + k * GB for k in (1, 2, 3, 4, 5))
    try:
        ol.ol_decode_step(ol.OL_LAYOUT_PAGED, desc, updated, q, Hkv * G, new_kv, np.array(lens, np.int32),
                          lens_dev, 0.0, -1, out, ol.OL_BF16, ws, ol.ol_workspace_size(B, Hkv * G, Hkv, D),
                          stream=0)
        status = ol.OL_OK
    except ol.OlError as e:
        status = e.status
    assert status == want, (case, status)


# the integer ranges of the affine formats (QuantizeLinear's output types)
AFFINE_RANGE = {ol.OL_FMT_I8: (-128, 127), ol.OL_FMT_U8: (0, 255), ol.OL_FMT_I4: (-8, 7), ol.OL_FMT_U4: (0, 15),
                ol.OL_FMT_I2: (-2, 1), ol.OL_FMT_U2: (0, 3)}
FLOAT_FORMATS = (ol.OL_FMT_F32, ol.OL_FMT_F16, ol.OL_FMT_BF16)


@st.composite
def plane_formats(draw):
    f = draw(st.integers(-1, 9))
    scale = draw(st.sampled_from([0.0, -0.5, float("inf"), float("nan"), 1e-30, 0.03125, 0.5, 3.0]))
    zp = draw(st.integers(-300, 300))
    return f, scale, zp


def plane_ok(f, scale, zp):
    if f in FLOAT_FORMATS:
        return True                                   # scale and zero point unused
    if f not in AFFINE_RANGE:
        return False
    lo, hi = AFFINE_RANGE[f]
    return scale > 0 and np.isfinite(scale) and lo <= zp <= hi


@settings(max_examples=400, deadline=None, derandomize=True)
@given(plane_formats(), plane_formats())
def test_page_format_rules(kf, vf):
    # the formats a heterogeneous append starts its pages in: a known format;
    # for the affine ones a positive finite scale and a zero point inside the
    # format's integer range
    B, H, S, M, D = 2, 2, 16, 8, 128
    P = B * M
    mirror = np.zeros(P, ol.PAGE_FORMAT_DTYPE)
    mirror["kf"], mirror["ks"], mirror["vf"], mirror["vs"] = ol.OL_FMT_BF16, 1.0, ol.OL_FMT_BF16, 1.0
    pool, fmt_dev, bt = BASE, BASE + 7 * GB, BASE + 8 * GB
    kv = ol.hpaged_kv(pool, fmt_dev, mirror, bt, np.arange(P, dtype=np.int32).reshape(B, M), kv_heads=H,
                      page_size=S, head_dim=D)
    fmt = ol.page_format(k=kf, v=vf)
    pos = np.array([0, 3 * S], np.int32)           # both rows start a page
    try:
        ol.ol_hpaged_append(kv, pool, BASE + GB, 1, pos, BASE + 2 * GB, fmt, stream=0)
        status = ol.OL_OK
    except ol.OlError as e:
        status = e.status
    want = ol.OL_ERR_INJECTED if plane_ok(*kf) and plane_ok(*vf) else ol.OL_ERR_SHAPE
    assert status == want, (kf, vf, status)
