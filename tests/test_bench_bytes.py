"""The algorithmic bytes behind every roofline figure of bench.py, checked
against an independent count on small workloads: the bytes of every K/V
element of every attended token in its storage format, the block-table and
page-format entries a paged step reads, the appended token(s) read and
written, q read and y written. Also the shape of the JSON fields per_config
carries. CPU only."""
import numpy as np

import bench
from workloads import AGE_FORMATS, Workload, page_format_classes

BITS = {0: 32, 1: 16, 2: 16, 3: 8, 4: 8, 5: 4, 6: 4, 7: 2, 8: 2}


def count(w, lens):
    """Token by token: what a step reads and writes (history rows = lens - T)."""
    T, D, H, Hq = w.chunk, w.head_dim, w.kv_heads, w.q_heads
    total = 0
    for b, n in enumerate(lens):
        hist = int(n) - T
        for t in range(hist):
            for _ in range(H):
                if w.layout == "int4":
                    total += 2 * (D // 2 + 2 * (D // 32) + D // 64)       # codes, fp16 scales, zero points; K and V
                elif w.layout == "hpaged":
                    (k, v) = AGE_FORMATS[page_format_classes(lens, w.page_size, w.max_pages_per_row)[b, t // w.page_size]][1]
                    total += D * (BITS[k[0]] + BITS[v[0]]) // 8
                else:
                    total += 2 * D * (2 if w.dtype == "bf16" else 4)
        if w.layout in ("paged", "hpaged"):
            pages = -(-int(n) // w.page_size)
            total += pages * (4 if w.layout == "paged" else 4 + 24)          # block-table entries (+ format pairs)
        for _ in range(T * H):
            if w.layout == "int4":
                total += 2 * D * 2 + 2 * (D // 2 + 2 * (D // 32) + D // 64)  # new K/V read (bf16), written encoded
            elif w.layout == "hpaged":
                (k, v) = AGE_FORMATS[0][1]
                total += 2 * D * 2 + D * (BITS[k[0]] + BITS[v[0]]) // 8
            else:
                e = 2 if w.dtype == "bf16" else 4
                total += 2 * 2 * D * e                                      # new K/V read and written
        total += 2 * Hq * T * D * 2                                         # q read, y written (bf16)
    return total


def test_step_bytes_match_an_independent_count():
    rng = np.random.default_rng(5)
    cases = [
        Workload("c", "bf16", 3, 8, 2, 64, 64, "contiguous", seed=1),
        Workload("p", "bf16", 3, 8, 2, 64, 64, "paged", seed=1, page_size=16, num_pages=32),
        Workload("i", "bf16", 3, 8, 2, 64, 64, "int4", seed=1),
        Workload("h", "bf16", 3, 8, 2, 64, 64 * 40, "hpaged", seed=1, page_size=16, num_pages=600),
        Workload("cc", "bf16", 3, 8, 2, 64, 64, "contiguous", seed=1, chunk=3),
        Workload("ic", "bf16", 3, 8, 2, 64, 64, "int4", seed=1, chunk=3),
        Workload("hc", "bf16", 3, 8, 2, 64, 64 * 40, "hpaged", seed=1, page_size=16, num_pages=600, chunk=3),
    ]
    for w in cases:
        hi = 64 if w.layout != "hpaged" else 64 * 40
        lens = rng.integers(w.chunk, hi + 1, size=w.batch).astype(np.int32)
        assert bench.step_bytes(w, lens) == count(w, lens), w.name


def test_compact_carries_the_per_config_fields():
    r = {"value": 1.0, "us_per_step": 2.0, "steps": 20,
         "us_per_step_spread": {"p10": 1.9, "median": 2.0, "p90": 2.1},
         "roofline": {"frac": 0.5, "traffic": 10}, "config": {"bytes_per_step": 4.0}, "rows_tok_per_s": 3.0,
         "gpu_launches": 20, "device_status": 0, "clocks": {"sm_mhz": 2070.0, "reasons": []},
         "e2e": {"us_per_step": 2.5}, "cpu_baseline": {"value": 0.1, "cores": 16, "us_per_step": 9.0,
                                                          "single_core": {"us_per_step": 90.0}}}
    c = bench.compact(r)
    assert c["spread_us"] == [1.9, 2.0, 2.1] and c["frac"] == 0.5 and c["traffic"] == 10
    assert c["clocks"] == [2070.0, []] and c["e2e_us_per_step"] == 2.5
    assert c["cpu_baseline"] == {"value": 0.1, "cores": 16, "us_per_step": 9.0, "one_core_us": 90.0}


def test_recorded_traffic_only_for_the_recorded_workload_and_sources():
    """A traffic figure belongs to one full-size workload on one version of its
    kernel sources: every line of the record resolves on the current sources,
    and a reduced copy of the same workload (--rows) gets none."""
    for name in ("qwen_b1_gqa7", "paged_b64", "int4_b16", "hpaged_b64"):
        w = bench.workload_of(name)
        t = bench.recorded_traffic(w)
        assert t is not None and t > 0, name
        if w.batch > 1:
            assert bench.recorded_traffic(bench.workload_of(name, w.batch // 2)) is None, name
