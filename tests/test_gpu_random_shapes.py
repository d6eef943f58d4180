"""Seeded random sweeps of the fused decode step on the GPU against the CPU
oracle: contiguous caches and paged pools with drawn batch, kv heads, query
group (1-8, the tensor-core range), head_dim (128, and 64 on the CUDA-core
kernel), capacity or page geometry, ragged lengths (1 and the full capacity
included), windows and the history-stable access bit. The planner picks the
kernel variant, cluster size, split count and launch order per shape, so the
sweep reaches combinations the hand-picked shapes do not. Every cache byte
must match the oracle's append and every output the oracle's attention within
the tolerance of the other parity tests. The INT4 and heterogeneous-page
sweeps do the same for those layouts (codes, scales, zero points, page
formats bit-exact).
"""
import numpy as np
import pytest

import oracle as O
import place_kv_cache_gb300 as ol
from workloads import Workload, bf16_from_f32, block_table, contiguous_cache, make_case, poisoned_pool
from tests.gpu_util import check_out, out_as_f64, out_tensor, to_dev, to_host, workspace

pytestmark = pytest.mark.gpu


def draw_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        layout = "paged" if rng.integers(2) else "contiguous"
        B = int(rng.integers(1, 7))
        Hkv = int(rng.integers(1, 9))
        G = int(rng.integers(1, 9))
        D = 128 if rng.random() < 0.85 else 64
        window = int(rng.choice([-1, -1, 0, 1, 15, 100]))
        stable = bool(rng.integers(2))
        if layout == "contiguous":
            C = int(rng.integers(16, 2049))
            S = M = P = 0
        else:
            S = int(rng.choice([16, 32]))
            M = int(rng.integers(1, 65))
            C = S * M
            P = B * M + int(rng.integers(0, 32))
        lens = rng.integers(1, C + 1, size=B)
        if B > 1:                      # edge rows: a single token, and a full row
            lens[int(rng.integers(B))] = 1
            lens[int(rng.integers(B))] = C
        cases.append(dict(id=f"{i:02d}-{layout}-B{B}-H{Hkv}x{G}-D{D}-C{C}-w{window}{'-stable' if stable else ''}",
                          layout=layout, B=B, Hkv=Hkv, G=G, D=D, C=C, S=S, M=M, P=P,
                          lens=lens.astype(np.int32), window=window, stable=stable, seed=int(rng.integers(1 << 30))))
    return cases


CASES = draw_cases(48, 2026)


@pytest.mark.parametrize("c", CASES, ids=[c["id"] for c in CASES])
def test_random_shape_fused_step(c):
    B, Hkv, G, D, C, lens, window = c["B"], c["Hkv"], c["G"], c["D"], c["C"], c["lens"], c["window"]
    Hq = Hkv * G
    access = ol.OL_READ_WRITE | (ol.OL_HISTORY_STABLE if c["stable"] else 0)
    ws, n = workspace(B, Hq, Hkv, D)
    out = out_tensor(B, Hq, D, ol.OL_BF16)
    if c["layout"] == "contiguous":
        w = Workload("rnd", "bf16", B, Hq, Hkv, D, C, "contiguous", seed=c["seed"])
        case = make_case(w, lens=lens)
        cache = contiguous_cache(case)
        cache_d = to_dev(cache)
        ol.ol_decode_step(ol.OL_LAYOUT_CONTIGUOUS, ol.kv_cache(cache_d, access=access), cache_d, to_dev(case.q), Hq,
                          to_dev(case.new_kv), lens, to_dev(lens), 0.0, window, out, ol.OL_BF16, ws, n)
        got = out_as_f64(out)
        O.cache_update(cache, case.new_kv, lens - 1)
        np.testing.assert_array_equal(to_host(cache_d), cache)
        want = O.decode_attention(case.q, cache, lens, window=window)
    else:
        w = Workload("rnd", "bf16", B, Hq, Hkv, D, C, "paged", seed=c["seed"], page_size=c["S"], num_pages=c["P"],
                     lens_range=(1, C))
        case = make_case(w, lens=lens)
        table = block_table(case)
        pool = poisoned_pool(w)
        for b, h in enumerate(case.history):
            if h.shape[2]:
                O.paged_update(pool, table[b:b + 1], h[:, None], [0])
        pool_d = to_dev(pool)
        desc = ol.paged_kv(pool_d, to_dev(table), table, access=access)
        ol.ol_decode_step(ol.OL_LAYOUT_PAGED, desc, pool_d, to_dev(case.q), Hq, to_dev(case.new_kv), lens,
                          to_dev(lens), 0.0, window, out, ol.OL_BF16, ws, n)
        got = out_as_f64(out)
        O.paged_update(pool, table, case.new_kv, lens - 1)
        np.testing.assert_array_equal(to_host(pool_d), pool)
        want = O.paged_attention(case.q, pool, table, lens, window=window)
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    check_out(got, want, ol.OL_BF16)


def draw_int4_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        B = int(rng.integers(1, 7))
        Hkv = int(rng.integers(1, 9))
        G = int(rng.integers(1, 9))
        D = 128 if rng.random() < 0.8 else 64
        C = int(rng.integers(16, 1501))
        window = int(rng.choice([-1, -1, 0, 3, 40]))
        mode = O.Q_FIXED if rng.random() < 0.3 else O.Q_DYNAMIC
        lens = rng.integers(1, C + 1, size=B)
        if B > 1:
            lens[int(rng.integers(B))] = 1
            lens[int(rng.integers(B))] = C
        cases.append(dict(id=f"{i:02d}-int4-B{B}-H{Hkv}x{G}-D{D}-C{C}-w{window}-{'fixed' if mode == O.Q_FIXED else 'dyn'}",
                          B=B, Hkv=Hkv, G=G, D=D, C=C, lens=lens.astype(np.int32), window=window, mode=mode,
                          seed=int(rng.integers(1 << 30))))
    return cases


INT4_CASES = draw_int4_cases(24, 2027)


@pytest.mark.parametrize("c", INT4_CASES, ids=[c["id"] for c in INT4_CASES])
def test_random_shape_int4_step(c):
    # the fused INT4 step: the new token quantized into the planes (bit-exact
    # with the oracle's encoding), history attended from the codes, the
    # current token uncompressed
    B, Hkv, G, D, C, lens, window, mode = c["B"], c["Hkv"], c["G"], c["D"], c["C"], c["lens"], c["window"], c["mode"]
    Hq = Hkv * G
    w = Workload("rnd4", "bf16", B, Hq, Hkv, D, C, "int4", seed=c["seed"])
    case = make_case(w, lens=lens)
    planes = O.int4_planes(B, Hkv, C, D)
    for b, h in enumerate(case.history):
        if h.shape[2]:
            sub = O.int4_planes(1, Hkv, C, D)
            O.int4_append(*sub, h[:, None], [0], mode=mode)
            for full, part in zip(planes, sub):
                full[:, b] = part[:, 0]
    dplanes = tuple(to_dev(p) for p in planes)
    ws, n = workspace(B, Hq, Hkv, D)
    out = out_tensor(B, Hq, D, ol.OL_F32)
    ol.ol_decode_step(ol.OL_LAYOUT_INT4, ol.int4_kv(*dplanes, head_dim=D, quant_mode=mode), dplanes[0],
                      to_dev(case.q), Hq, to_dev(case.new_kv), lens, to_dev(lens), 0.0, window, out, ol.OL_F32,
                      ws, n)
    got = out_as_f64(out)
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    O.int4_append(*planes, case.new_kv, lens - 1, mode=mode)
    for g, r in zip((to_host(p) for p in dplanes), planes):
        np.testing.assert_array_equal(g, r)
    want = O.int4_attention(case.q, *planes, lens, cur_kv=case.new_kv, window=window)
    check_out(got, want, ol.OL_F32)


def draw_hpaged_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        B = int(rng.integers(1, 5))
        H = int(rng.integers(1, 5))
        G = int(rng.integers(1, 9))
        S = int(rng.choice([16, 32]))
        D = 128 if rng.random() < 0.75 else 64
        M = int(rng.integers(1, 9))
        window = int(rng.choice([-1, -1, 0, 5, 40]))
        lens = rng.integers(1, M * S + 1, size=B)
        cases.append(dict(id=f"{i:02d}-hpaged-B{B}-H{H}x{G}-S{S}-D{D}-M{M}-w{window}", B=B, H=H, G=G, S=S, D=D, M=M,
                          lens=lens.astype(np.int32), window=window, seed=int(rng.integers(1 << 30))))
    return cases


HPAGED_CASES = draw_hpaged_cases(16, 2028)


@pytest.mark.parametrize("c", HPAGED_CASES, ids=[c["id"] for c in HPAGED_CASES])
def test_random_shape_hpaged_step(c):
    # history written page by page in drawn formats (every page its own K/V
    # formats), then one fused step whose new page (if it starts one) takes
    # the call's formats: pool bytes, format table and mirror bit-exact,
    # outputs against the oracle
    from tests.test_gpu_hpaged import FORMATS, Pair, fmt_pair
    B, H, G, S, D, M, lens, window = c["B"], c["H"], c["G"], c["S"], c["D"], c["M"], c["lens"], c["window"]
    Hq = H * G
    pr = Pair(B, H, S, D, M, B * M + 2, seed=c["seed"])
    pick = pr.rng.integers(0, len(FORMATS), size=(B, M))
    pr.fill(lens - 1, lambda b, j: int(pick[b, j]))
    q = bf16_from_f32(pr.rng.standard_normal((B, Hq, D)).astype(np.float32))
    new_kv = pr.values(1)
    od, gd = fmt_pair(int(pr.rng.integers(len(FORMATS))))
    want = O.hpaged_attention(q, pr.pool, pr.desc, pr.table, lens, H, cur_kv=new_kv, window=window)
    O.hpaged_append(pr.pool, pr.desc, pr.table, new_kv, lens - 1, od)
    ws, n = workspace(B, Hq, H, D)
    out = out_tensor(B, Hq, D, ol.OL_F32)
    ol.ol_hpaged_decode_step(pr.kv, pr.pool_d, to_dev(q), Hq, to_dev(new_kv), gd, lens, to_dev(lens), 0.0, window,
                             out, ol.OL_F32, ws, n)
    got = out_as_f64(out)
    assert ol.ol_workspace_status(ws) == ol.OL_DEVICE_OK
    pr.check_state()
    check_out(got, want, ol.OL_F32)
