"""Decode-step benchmark: achieved HBM GB/s (and % of the measured HBM
roofline), microseconds per step and rows x tokens / s of the fused decode
step (in-place append + GQA decode attention) over a caller-owned KV cache.

One step = one ``ol_decode_step`` over the whole batch of the workload: host
validation, the append of one token per row and attention over every row's
valid prefix, in one kernel launch (a chunked step: the append, then the
attention). Steps are replayed from CUDA graphs so the host never limits a
microsecond-scale step; when one step's cache fits in L2, consecutive steps
rotate over enough independent cache replicas that the data of a step is never
L2-resident from the previous visit.

Without --workload the headline line is the paged pool of 64 rows (the largest
workload that fits one GPU) and ``per_config`` carries the same figures for
every other workload: the single-row GQA-7 step, the ragged batch of 32 rows,
the INT4 cache over its 64-step chain, the chunked step of 4 tokens and the
heterogeneous pages. Every workload times exactly --steps steps (a chained
workload at least its whole chain).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                       [--impl ours|reference]
Under torchrun each rank runs its own replica of the workload on its own GPU
(independent rows: no collective on the data path; weak scaling); rank 0
prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import AGE_FORMATS, WORKLOADS, bf16_from_f32, make_case, page_format_classes  # noqa: E402

FORMAT_BITS = {0: 32, 1: 16, 2: 16, 3: 8, 4: 8, 5: 4, 6: 4, 7: 2, 8: 2}   # heterogeneous page formats

METRIC = "decode step: achieved HBM GB/s (% of ~8 TB/s roofline), µs/step, rows·tok/s"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=None, choices=[k for k in WORKLOADS if k != "tiny_f32"],
                    help="one workload only (default: the headline workload and per_config for the others)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seconds", type=float, default=1.0, help="target timed seconds when --steps is not given")
    ap.add_argument("--phase-stamps", action="store_true",
                    help="timing build: per-CTA phase stamps of the decode kernel over one graph of steps")
    ap.add_argument("--phase-out", default=None, help="with --phase-stamps: save the raw stamps (.npy) here")
    ap.add_argument("--rows", type=int, default=None,
                    help="the workload's first ROWS rows only (a smaller device footprint, for profiling)")
    return ap.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# Device-code sources each layout's timed kernel is built from (the shared
# headers included): a recorded DRAM traffic figure holds only while these are
# unchanged.
_SHARED = ("ol_common.cuh", "ol_merge.cuh", "ol_internal.h")
KERNEL_SOURCES = {"contiguous": ("ol_fast_bf16.cu", "ol_fast_bf16_kernel.inc") + _SHARED,
                  "paged": ("ol_fast_bf16.cu", "ol_fast_bf16_kernel.inc") + _SHARED,
                  "int4": ("ol_fast_int4.cu",) + _SHARED,
                  "hpaged": ("ol_fast_hpaged.cu", "ol_hpaged.cuh") + _SHARED}


def kernel_sources_sha(layout: str) -> str:
    """sha256 over the device-code sources of a layout's kernel (file name and
    content, in name order)."""
    import hashlib
    d = os.path.join(ROOT, "place_kv_cache_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(KERNEL_SOURCES[layout]):
        h.update(name.encode() + b"\0")
        with open(os.path.join(d, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(w):
    """DRAM bytes (read + write) per launch of the workload's kernel from one ncu
    capture, as listed in profiles/dram_traffic.txt; None when none was recorded,
    it was recorded on other kernel sources, or the workload is a reduced copy
    (--rows) of the recorded one."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path) or WORKLOADS.get(w.name) != w:
        return None
    sha = kernel_sources_sha(w.layout)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 4 and not line.startswith("#") and parts[0] == w.name and parts[3] == sha:
                return int(parts[2])
    return None


def step_bytes(w, lens):
    """Algorithmic HBM bytes of one step: K/V of every attended token (the new
    token's K/V read from new_kv), the appended token written, q read, y written.
    A chunked step appends T = w.chunk tokens per row and reads the union of its
    query tokens' ranges once: history, the chunk's K/V, T queries and outputs."""
    elt = 2 if w.dtype == "bf16" else 4
    D = w.head_dim
    T = w.chunk
    if w.layout == "hpaged":
        # each history token in its page's formats (K and V rows of D * bits / 8
        # bytes), plus a block-table entry and a 24-byte format pair per page;
        # the T new tokens read uncompressed (bf16) and written in the format of
        # the pages they start (age 0); T queries and outputs
        S, M = w.page_size, w.max_pages_per_row
        cls = page_format_classes(lens, S, M)
        row = [D * (FORMAT_BITS[k[0]] + FORMAT_BITS[v[0]]) // 8 for _, (k, v) in AGE_FORMATS]
        hist = 0.0
        for b, n in enumerate(lens):
            h = int(n) - T
            for j in range((h + S - 1) // S):
                hist += min(S, h - j * S) * row[cls[b, j]]
        hist = hist * w.kv_heads + float(np.sum(np.ceil(lens / S))) * (4 + 24)
        cur = w.batch * w.kv_heads * T * 2 * D * 2
        written = w.batch * w.kv_heads * T * row[0]
        q = w.batch * w.q_heads * T * D * 2
        return hist + cur + written + q + q
    if T > 1 and w.layout == "int4":
        # history codes, scales and zero points; the chunk read uncompressed (bf16) and
        # written quantized; T queries and outputs
        kv_tok = 2 * (D // 2 + (D // 32) * 2 + D // 64)
        hist = float(np.sum(lens - T)) * w.kv_heads * kv_tok
        return hist + w.batch * w.kv_heads * T * (2 * D * 2 + kv_tok) + 2 * w.batch * w.q_heads * T * D * 2
    if T > 1:
        hist = float(np.sum(lens - T)) * w.kv_heads * 2 * D * elt
        new = w.batch * w.kv_heads * T * 2 * D * elt
        return hist + 2 * new + 2 * w.batch * w.q_heads * T * D * 2   # new K/V written and read; q and y
    if w.layout == "int4":
        kv_tok = 2 * (D // 2 + (D // 32) * 2 + D // 64)         # codes + fp16 scales + zero points, K and V
        hist = float(np.sum(lens - 1)) * w.kv_heads * kv_tok
        cur = w.batch * w.kv_heads * 2 * D * 2                   # current token read uncompressed (bf16)
        written = w.batch * w.kv_heads * kv_tok
    else:
        hist = float(np.sum(lens - 1)) * w.kv_heads * 2 * D * elt
        cur = w.batch * w.kv_heads * 2 * D * elt
        written = w.batch * w.kv_heads * 2 * D * elt
        if w.layout == "paged":
            hist += float(np.sum(np.ceil(lens / w.page_size))) * 4   # block-table entries
    q = w.batch * w.q_heads * D * 2
    y = w.batch * w.q_heads * D * 2
    return hist + cur + written + q + y


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- multi-rank

def combine_ranks(ms_total, steps, bytes_per_step, world, dist=None, device="cpu"):
    """Whole-job result of a weak-scaling run: every rank processes its own copy
    of the workload (independent rows: no collective on the data path); the job
    time is the slowest rank's (max over ranks) and the job moves world x the
    per-rank bytes. Returns (ms_per_step, whole-job GB/s)."""
    if dist is not None and world > 1:
        import torch
        t = torch.tensor([ms_total], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_total = float(t.item())
    ms_per_step = ms_total / steps
    return ms_per_step, bytes_per_step * world / (ms_per_step * 1e-3) / 1e9


# ------------------------------------------------------------------- ours

def to_dev(a, dev):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


class Setup:
    """Device-resident inputs for one workload (one rank)."""

    def __init__(self, w, dev, seed_offset=0):
        import torch
        import place_kv_cache_gb300 as ol
        self.ol, self.torch, self.w, self.dev = ol, torch, w, dev
        gen = torch.Generator(device=dev)
        gen.manual_seed(w.seed + 1000 * seed_offset)
        rng = np.random.default_rng(w.seed + 1000 * seed_offset)
        # lengths and page permutation from the seeded generator; bulk values from a seeded
        # device generator (N(0,1), rounded to bf16): the benchmark times the path, the tests
        # check its values against the oracle
        from workloads import draw_lens
        self.lens = draw_lens(rng, w)
        # a chained workload advances every row by one token per step (append at
        # lens - 1, lens + 1 next step); the others repeat the same step shape
        self.chain = w.steps if w.steps > 1 else 1
        self.lens_list = [self.lens + i for i in range(self.chain)]
        self.lens_d_list = [torch.from_numpy(l).to(dev) for l in self.lens_list]
        self.lens_d = self.lens_d_list[0]
        D = w.head_dim
        B, H = w.batch, w.kv_heads
        self.bytes_per_step = float(np.mean([step_bytes(w, l) for l in self.lens_list]))
        T = w.chunk
        qshape = (B, w.q_heads, T, D) if T > 1 else (B, w.q_heads, D)
        self.q = torch.randn(qshape, generator=gen, device=dev).to(torch.bfloat16)
        self.new_kv = torch.randn((2, B, H, T, D), generator=gen, device=dev).to(torch.bfloat16)
        self.out = torch.empty(qshape, dtype=torch.bfloat16, device=dev)
        ws_bytes = (ol.ol_workspace_size_chunk(B, w.q_heads, H, D, T) if T > 1 else
                    ol.ol_workspace_size(B, w.q_heads, H, D))
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        self.ws_bytes = ws_bytes
        ol.ol_workspace_init(self.ws, ws_bytes)
        self.replicas = max(1, math.ceil(2 * L2_BYTES / max(1.0, self.bytes_per_step)))
        self.replicas = min(self.replicas, 64)
        self.caches, self.descs, self.updated = [], [], []
        for r in range(self.replicas):
            self._make_replica(gen, rng)
        self.l2_note = (f"{self.replicas} cache replicas rotated, {self.replicas * self.bytes_per_step / 2**20:.0f} MiB "
                        f"touched per rotation > 2x L2" if self.replicas > 1 else
                        f"inputs larger than L2 ({self.bytes_per_step / 2**20:.0f} MiB per step)")

    def resident_bytes(self):
        w = self.w
        if w.layout == "paged":
            return 2 * w.num_pages * w.kv_heads * w.page_size * w.head_dim * 2
        if w.layout == "hpaged":
            return 2 * w.num_pages * w.kv_heads * w.page_size * w.head_dim * 4
        if w.layout == "int4":
            return 2 * w.batch * w.kv_heads * w.capacity * (w.head_dim // 2 + w.head_dim // 16 + w.head_dim // 64)
        return 2 * w.batch * w.kv_heads * w.capacity * w.head_dim * 2

    def _make_replica(self, gen, rng):
        torch, ol, w = self.torch, self.ol, self.w
        B, H, D = w.batch, w.kv_heads, w.head_dim
        # consecutive steps either use other caches (replicas, like the layers of
        # a model) or rewrite only their own new row: the history is stable and
        # the first tiles may be requested before the previous step completes.
        # A chained workload appends where the next step reads: no such promise.
        acc = ol.OL_READ_WRITE | (ol.OL_HISTORY_STABLE if self.chain == 1 else 0)
        if w.layout == "contiguous":
            cache = torch.randn((2, B, H, w.capacity, D), generator=gen, device=self.dev).to(torch.bfloat16)
            self.caches.append(cache)
            self.descs.append(ol.kv_cache(cache, access=acc))
            self.updated.append(cache)
            self.layout = ol.OL_LAYOUT_CONTIGUOUS
        elif w.layout == "paged":
            pool = torch.empty((2, w.num_pages, H, w.page_size, D), dtype=torch.bfloat16, device=self.dev)
            for k in range(2):
                for c0 in range(0, w.num_pages, 4096):
                    c1 = min(w.num_pages, c0 + 4096)
                    pool[k, c0:c1] = torch.randn((c1 - c0, H, w.page_size, D), generator=gen,
                                                 device=self.dev).to(torch.bfloat16)
            perm = rng.permutation(w.num_pages).astype(np.int32)
            M = w.max_pages_per_row
            table = np.ascontiguousarray(perm[: B * M].reshape(B, M))
            bt_d = torch.from_numpy(table).to(self.dev)
            self.caches.append((pool, bt_d, table))
            self.descs.append(ol.paged_kv(pool, bt_d, table, access=acc))
            self.updated.append(pool)
            self.layout = ol.OL_LAYOUT_PAGED
        elif w.layout == "hpaged":
            self._make_hpaged_replica(gen, rng, acc)
        else:
            rows = 2 * B * H * w.capacity
            codes = torch.randint(0, 256, (2, B, H, w.capacity, D // 2), generator=gen, device=self.dev,
                                  dtype=torch.int32).to(torch.uint8)
            scales = (torch.rand((2, B, H, w.capacity, D // 32), generator=gen, device=self.dev) * 0.3 + 0.05)
            scales = scales.to(torch.float16).view(torch.int16)
            zps = torch.randint(0, 256, (2, B, H, w.capacity, D // 64), generator=gen, device=self.dev,
                                dtype=torch.int32).to(torch.uint8)
            del rows
            self.caches.append((codes, scales, zps))
            self.descs.append(ol.int4_kv(codes, scales, zps, head_dim=D, access=acc))
            self.updated.append(codes)
            self.layout = ol.OL_LAYOUT_INT4

    def _make_hpaged_replica(self, gen, rng, acc):
        """Every row's history (lens - 1 tokens) appended through the library in
        the formats of its pages' ages: one append per run of pages of one class."""
        torch, ol, w = self.torch, self.ol, self.w
        B, H, D, S, M, P = w.batch, w.kv_heads, w.head_dim, w.page_size, w.max_pages_per_row, w.num_pages
        pool = torch.empty(P * 2 * H * S * D * 4, dtype=torch.uint8, device=self.dev)
        mirror = np.zeros(P, ol.PAGE_FORMAT_DTYPE)
        (kf, ks, kz), (vf, vs, vz) = AGE_FORMATS[0][1]
        mirror["kf"], mirror["ks"], mirror["kz"], mirror["vf"], mirror["vs"], mirror["vz"] = kf, ks, kz, vf, vs, vz
        fmt_d = torch.from_numpy(mirror.view(np.uint8).copy()).to(self.dev)
        perm = rng.permutation(P).astype(np.int32)
        table = np.ascontiguousarray(perm[: B * M].reshape(B, M))
        bt_d = torch.from_numpy(table).to(self.dev)
        cls = page_format_classes(self.lens, S, M)
        for b in range(B):
            hist = int(self.lens[b]) - w.chunk
            row_t = np.ascontiguousarray(table[b:b + 1])
            row_kv = ol.hpaged_kv(pool, fmt_d, mirror, bt_d[b:b + 1], row_t, kv_heads=H, page_size=S, head_dim=D)
            j = 0
            npages = (hist + S - 1) // S
            while j < npages:
                j1 = j
                while j1 < npages and cls[b, j1] == cls[b, j]:
                    j1 += 1
                t0, t1 = j * S, min(j1 * S, hist)
                vals = torch.randn((2, 1, H, t1 - t0, D), generator=gen, device=self.dev).to(torch.bfloat16)
                k, v = AGE_FORMATS[cls[b, j]][1]
                pos = np.array([t0], np.int32)
                ol.ol_hpaged_append(row_kv, pool, vals, t1 - t0, pos, torch.from_numpy(pos).to(self.dev),
                                    ol.page_format(k=k, v=v))
                j = j1
        torch.cuda.synchronize()
        self.new_pages = ol.page_format(*AGE_FORMATS[0][1])
        self.caches.append((pool, fmt_d, mirror, bt_d, table))
        self.descs.append(ol.hpaged_kv(pool, fmt_d, mirror, bt_d, table, kv_heads=H, page_size=S, head_dim=D,
                                       access=acc))
        self.updated.append(pool)
        self.layout = ol.OL_LAYOUT_HPAGED

    def step(self, i, stream=None):
        """Step i of the rotation: replica i % replicas, chain position i % chain."""
        r, c = i % self.replicas, i % self.chain
        if self.w.chunk > 1 and self.w.layout == "hpaged":
            self.ol.ol_hpaged_chunk_step(self.descs[r], self.updated[r], self.q, self.w.q_heads, self.w.chunk,
                                         self.new_kv, self.new_pages, self.lens_list[c], self.lens_d_list[c], 0.0, -1,
                                         self.out, self.ol.OL_BF16, self.ws, self.ws_bytes, stream=stream)
            return
        if self.w.chunk > 1:
            self.ol.ol_chunk_step(self.layout, self.descs[r], self.updated[r], self.q, self.w.q_heads, self.w.chunk,
                                  self.new_kv, self.lens_list[c], self.lens_d_list[c], 0.0, -1, self.out,
                                  self.ol.OL_BF16, self.ws, self.ws_bytes, stream=stream)
            return
        if self.w.layout == "hpaged":
            self.ol.ol_hpaged_decode_step(self.descs[r], self.updated[r], self.q, self.w.q_heads, self.new_kv,
                                          self.new_pages, self.lens_list[c], self.lens_d_list[c], 0.0, -1, self.out,
                                          self.ol.OL_BF16, self.ws, self.ws_bytes, stream=stream)
            return
        self.ol.ol_decode_step(self.layout, self.descs[r], self.updated[r], self.q, self.w.q_heads, self.new_kv,
                               self.lens_list[c], self.lens_d_list[c], 0.0, -1, self.out, self.ol.OL_BF16, self.ws,
                               self.ws_bytes, stream=stream)


# ------------------------------------------------------------- driver

# The headline workload is the largest one that fits one GPU (the paged pool of
# 64 rows); every other workload is measured in the same run under per_config.
HEADLINE = "paged_b64"
PER_CONFIG = ("qwen_b1_gqa7", "ragged_b32", "int4_b16", "chunk4_b32", "int4chunk4_b16", "hpaged_b64",
              "hpchunk4_b64")
# oracle samples cut to fewer rows where the oracle's own composition is slow
# (the INT4 chunked attention decodes the history row by row in Python)
ORACLE_ROWS = {"int4chunk4_b16": 2, "hpchunk4_b64": 2}


def workload_of(name, rows=None):
    """The named workload, or its first `rows` rows (pages sized to those rows)."""
    from workloads import scaled
    w = WORKLOADS[name]
    if rows is not None and rows < w.batch:
        w = scaled(w, batch=rows)
        if w.layout in ("paged", "hpaged"):
            w = scaled(w, num_pages=rows * w.max_pages_per_row)
    return w


def launches_per_step(w) -> int:
    """Kernel launches of one step: a chunked step appends and attends in two
    launches; a decode step is one fused launch."""
    return 2 if w.chunk > 1 else 1


def measure(w, args, rank, world, dist, dev, K_req):
    """Time exactly K_req steps of workload w (K_req None: about --seconds).

    Steps are replayed from CUDA graphs: full graphs of `per_graph` steps (a
    whole number of cache-replica rotations and chain positions) and, for the
    remainder, one graph of the first K mod per_graph steps of the rotation, so
    the timed region holds exactly K steps. The region is bracketed by a
    barrier and a stream synchronize on both sides and timed with CUDA events
    on the launching stream. The spread comes from further full graphs timed
    one by one after the region."""
    import torch
    s = Setup(w, dev, seed_offset=rank)
    stream = torch.cuda.Stream(device=dev)
    unit = s.replicas * s.chain
    per_graph = -(-max(unit, 32) // unit) * unit

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                s.step(i)
        return g

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3) * unit):
            s.step(i)
        stream.synchronize()
        g_full = capture(per_graph)
        g_full.replay()
        stream.synchronize()
    t = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(5):
            g_full.replay()
    stream.synchronize()
    est = (time.perf_counter() - t) / (5 * per_graph)
    K = K_req if K_req is not None else max(per_graph, int(args.seconds / max(est, 1e-7)) // per_graph * per_graph)
    n_full, rem = divmod(K, per_graph)
    g_tail = None
    if rem:
        with torch.cuda.stream(stream):
            g_tail = capture(rem)
            g_tail.replay()
            stream.synchronize()
    local = int(os.environ.get("LOCAL_RANK", 0))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    n_sp = max(5, min(50, int(0.3 / max(est * per_graph, 1e-7))))
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(n_sp + 1)]
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            for _ in range(max(1, int(0.3 / max(est * per_graph, 1e-7)))):
                g_full.replay()                  # keep the GPU busy while the sampler settles
        if dist is not None:
            dist.barrier()
        stream.synchronize()
        clk.mark_start()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n_full):
                g_full.replay()
            if g_tail is not None:
                g_tail.replay()
            e1.record(stream)
        stream.synchronize()
        clk.mark_end()
        if dist is not None:
            dist.barrier()
        with torch.cuda.stream(stream):            # spread: full graphs timed one by one
            marks[0].record(stream)
            for k in range(n_sp):
                g_full.replay()
                marks[k + 1].record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1)
    per_us = sorted(marks[k].elapsed_time(marks[k + 1]) * 1e3 / per_graph for k in range(n_sp))
    ms_per_step, gbs = combine_ranks(ms, K, s.bytes_per_step, world, dist, device=dev)
    import place_kv_cache_gb300 as ol
    status = ol.ol_workspace_status(s.ws, stream=stream)
    peak, peak_src = measured_peaks()
    frac = gbs / world / peak
    res = {
        "value": round(gbs, 2), "unit": "GB/s", "steps": K, "ms_per_step": ms_per_step,
        "us_per_step": round(ms_per_step * 1e3, 3),
        "us_per_step_spread": {"p10": round(float(np.percentile(per_us, 10)), 3),
                               "median": round(float(np.percentile(per_us, 50)), 3),
                               "p90": round(float(np.percentile(per_us, 90)), 3),
                               "graphs": n_sp, "graph_steps": per_graph},
        "rows_tok_per_s": round(w.batch * w.chunk * world / (ms_per_step * 1e-3), 1),
        "pct_of_hbm_roofline": round(100.0 * frac, 2),
        "dtype": {"int4": "u4+bf16", "hpaged": "bf16+i8+i4/u4 pages, f32 math"}.get(w.layout, "bf16"),
        "config": {"workload": w.name, "layout": w.layout, "batch": w.batch, "q_heads": w.q_heads,
                   "kv_heads": w.kv_heads, "head_dim": w.head_dim, "capacity": w.capacity,
                   "lens_mean": float(np.mean(s.lens)), "bytes_per_step": s.bytes_per_step, "l2": s.l2_note,
                   "graph_steps": per_graph, "tail_graph_steps": rem, "chained_steps": s.chain,
                   "history_stable": s.chain == 1, "parallelism": f"rows x{world} (independent)"},
        "roofline": {"bound": "hbm", "achieved": round(gbs / world, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(frac, 4), "traffic": recorded_traffic(w),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else
                     "fallback 6.8 TB/s"},
        "gpu_launches": K * launches_per_step(w),
        "device_status": status,
        "clocks": clk.summary(),
    }
    if w.chunk > 1:
        res["config"]["chunk"] = w.chunk
    if not args.no_e2e and w.chunk == 1 and w.layout != "hpaged":
        res["e2e"] = run_e2e(s, stream, K)
    elif not args.no_e2e:
        # the host-buffer call serves the decode step of the uniform layouts;
        # chunked steps and heterogeneous pages run from device buffers
        res["e2e"] = None
    del s, g_full, g_tail
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def compact(r):
    """The per-workload figures of a measure() result, for per_config: CUDA-event
    time of exactly `steps` steps, the spread over further graphs (p10, median,
    p90), roofline fraction and recorded DRAM traffic, clocks, the host-buffer
    time, and the oracle's time on the host cores."""
    out = {"value": r["value"], "us_per_step": r["us_per_step"], "steps": r["steps"],
           "spread_us": [r["us_per_step_spread"][k] for k in ("p10", "median", "p90")],
           "frac": r["roofline"]["frac"], "traffic": r["roofline"]["traffic"],
           "bytes_per_step": r["config"]["bytes_per_step"], "rows_tok_per_s": r["rows_tok_per_s"],
           "gpu_launches": r["gpu_launches"], "device_status": r["device_status"],
           "clocks": [r["clocks"]["sm_mhz"], r["clocks"]["reasons"]]}
    e = r.get("e2e")
    out["e2e_us_per_step"] = e["us_per_step"] if e else None
    cb = r.get("cpu_baseline")
    if cb:
        out["cpu_baseline"] = {"value": cb["value"], "cores": cb["cores"], "us_per_step": cb["us_per_step"],
                               "one_core_us": cb["single_core"]["us_per_step"]}
    return out


def run_e2e(s, stream, K_e2e):
    """The same step through the public host-buffer call, ol_decode_step_host:
    every step moves q and the new K/V from pinned host memory to the device
    (and the lengths when the launch cannot carry them by value), runs the step
    on the device-resident cache and moves y back into pinned host memory, all
    enqueued by that one call on the timed stream. Pinned buffers are mapped
    into the device's address space, so the step's kernels load the inputs and
    store y across the CPU-GPU link themselves (no copy-engine copies)."""
    torch, ol, w = s.torch, s.ol, s.w
    q_h = s.q.cpu().pin_memory()
    kv_h = s.new_kv.cpu().pin_memory()
    y_h = torch.empty(s.out.shape, dtype=s.out.dtype).pin_memory()
    lens_h = [torch.from_numpy(np.ascontiguousarray(l, dtype=np.int32)) for l in s.lens_list]  # host int32
    h2d = q_h.numel() * 2 + kv_h.numel() * 2 + (s.lens.size * 4 if w.batch > 160 else 0)
    d2h = y_h.numel() * 2
    n = ol.ol_workspace_size_host(w.batch, w.q_heads, w.kv_heads, w.head_dim)
    ws = torch.empty(n, dtype=torch.uint8, device=s.dev)
    ol.ol_workspace_init(ws, n)
    R = s.replicas
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def one(i):
        r, c = i % R, i % s.chain
        ol.ol_decode_step_host(s.layout, s.descs[r], s.updated[r], q_h, w.q_heads, kv_h, lens_h[c], 0.0, -1, y_h,
                               ol.OL_BF16, ws, n, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(3 * R * s.chain):
            one(i)
        stream.synchronize()
        e0.record(stream)
        for i in range(K_e2e):
            one(i)
        e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / K_e2e
    return {"value": round(s.bytes_per_step / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "us_per_step": round(ms * 1e3, 3),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": K_e2e,
            "call": "ol_decode_step_host per step; q, new K/V read and y written by its kernels in mapped pinned "
                    "host memory"}


# --------------------------------------------------------------- oracle

def host_threads() -> int:
    """Host cores this process may run on (at most 32)."""
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(n, 32))


def oracle_units(w, n_threads):
    """A bounded sample of the workload for the CPU oracle, cut into independent
    units of one step (append + attention), one per host thread: the first
    min(batch, n_threads) rows, a unit per row; a single-row workload is cut by
    kv head instead. Every unit works on its own arrays (or, for the paged
    pools, on its own row's pages of one shared pool), so the units of a step
    run side by side. Returns (units, sample workload, bytes of one step of the
    whole sample, description)."""
    import oracle as O
    from workloads import block_table, contiguous_cache, poisoned_pool, scaled
    by_head = w.batch == 1
    rows = 1 if by_head else min(w.batch, n_threads, ORACLE_ROWS.get(w.name, w.batch))
    ws = scaled(w, batch=rows)
    if w.layout in ("paged", "hpaged"):
        ws = scaled(ws, num_pages=rows * w.max_pages_per_row)
    T = w.chunk
    case = make_case(ws, seed=w.seed, history_len_offset=T)
    lens = case.lens
    H, G, D = ws.kv_heads, ws.group, ws.head_dim
    units = []
    if T > 1:
        rng = np.random.default_rng(w.seed + 7)
        q = bf16_from_f32(rng.standard_normal((rows, ws.q_heads, T, D)).astype(np.float32))
        kv = bf16_from_f32(rng.standard_normal((2, rows, H, T, D)).astype(np.float32))
    else:
        q, kv = case.q, case.new_kv
    # (row, kv heads) pieces: a row, or one kv head of the single row
    pieces = [(0, g) for g in range(H)] if by_head else [(b, None) for b in range(rows)]

    def sl_heads(a, g, axis):       # kv head g's slice along `axis` (None: all heads)
        if g is None:
            return a
        idx = [slice(None)] * a.ndim
        idx[axis] = slice(g, g + 1)
        return a[tuple(idx)]

    def sl_q(b, g):
        qb = q[b:b + 1]
        return np.ascontiguousarray(qb if g is None else qb[:, g * G:(g + 1) * G])

    def build(fn, items):          # per-unit set-up work on the host threads (the oracle is C)
        import concurrent.futures
        with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(items), n_threads))) as ex:
            return list(ex.map(fn, items))

    if w.layout == "contiguous":
        cache = contiguous_cache(case)
        for b, g in pieces:
            c = np.ascontiguousarray(sl_heads(cache[:, b:b + 1], g, 2))
            k = np.ascontiguousarray(sl_heads(kv[:, b:b + 1], g, 2))
            qq, lb = sl_q(b, g), np.ascontiguousarray(lens[b:b + 1])
            if T > 1:
                units.append(lambda c=c, k=k, qq=qq, lb=lb: (O.cache_update(c, k, lb - T),
                                                             O.chunk_attention(qq, c, lb, T)))
            else:
                units.append(lambda c=c, k=k, qq=qq, lb=lb: (O.cache_update(c, k, lb - 1),
                                                             O.decode_attention(qq, c, lb)))
        del cache
    elif w.layout == "int4" and T > 1:
        def quantized(b):
            planes = O.int4_planes(1, H, ws.capacity, D)
            O.int4_append(*planes, np.ascontiguousarray(case.history[b][:, None]), [0])
            return planes
        for b, planes in zip(range(rows), build(quantized, list(range(rows)))):
            k = np.ascontiguousarray(kv[:, b:b + 1])
            qq, lb = sl_q(b, None), np.ascontiguousarray(lens[b:b + 1])
            units.append(lambda pl=planes, k=k, qq=qq, lb=lb: (O.int4_chunk_attention(qq, *pl, lb, T, k),
                                                               O.int4_append(*pl, k, lb - T)))
    elif w.layout == "int4":
        def quantized(piece):
            b, g = piece
            hb = case.history[b] if g is None else case.history[b][:, g:g + 1]
            planes = O.int4_planes(1, hb.shape[1], ws.capacity, D)
            O.int4_append(*planes, np.ascontiguousarray(hb[:, None]), [0])
            return planes
        for (b, g), planes in zip(pieces, build(quantized, pieces)):
            k = np.ascontiguousarray(sl_heads(kv[:, b:b + 1], g, 2))
            qq, lb = sl_q(b, g), np.ascontiguousarray(lens[b:b + 1])
            units.append(lambda pl=planes, k=k, qq=qq, lb=lb: (O.int4_append(*pl, k, lb - 1),
                                                               O.int4_attention(qq, *pl, lb, cur_kv=k)))
    elif w.layout == "paged":
        pool = poisoned_pool(ws)
        table = block_table(case)

        def fill(b):               # rows own disjoint pages of the shared pool
            h = case.history[b]
            if h.shape[2]:
                O.paged_update(pool, table[b:b + 1], h[:, None], [0])
        build(fill, list(range(rows)))
        for b, _ in pieces:
            tb, k = np.ascontiguousarray(table[b:b + 1]), np.ascontiguousarray(kv[:, b:b + 1])
            qq, lb = sl_q(b, None), np.ascontiguousarray(lens[b:b + 1])
            units.append(lambda tb=tb, k=k, qq=qq, lb=lb: (O.paged_update(pool, tb, k, lb - 1),
                                                           O.paged_attention(qq, pool, tb, lb)))
    else:  # heterogeneous pages
        S, M = ws.page_size, ws.max_pages_per_row
        pool, desc = O.hpaged_pool(ws.num_pages, H, S, D)
        table = block_table(case)
        cls = page_format_classes(lens, S, M)

        def fill(b):               # one append per run of pages of one format class
            h = case.history[b]
            hist, j = h.shape[2], 0
            npages = (hist + S - 1) // S
            while j < npages:
                j1 = j
                while j1 < npages and cls[b, j1] == cls[b, j]:
                    j1 += 1
                kf, vf = AGE_FORMATS[cls[b, j]][1]
                O.hpaged_append(pool, desc, table[b:b + 1], h[:, None, :, j * S:min(j1 * S, hist)], [j * S],
                                O.page_desc(k=kf, v=vf))
                j = j1
        build(fill, list(range(rows)))
        new_fmt = O.page_desc(*AGE_FORMATS[0][1])
        for b, _ in pieces:
            tb, k = np.ascontiguousarray(table[b:b + 1]), np.ascontiguousarray(kv[:, b:b + 1])
            qq, lb = sl_q(b, None), np.ascontiguousarray(lens[b:b + 1])
            if T > 1:
                units.append(lambda tb=tb, k=k, qq=qq, lb=lb: (
                    O.hpaged_chunk_attention(qq, pool, desc, tb, lb, H, T, k),
                    O.hpaged_append(pool, desc, tb, k, lb - T, new_fmt)))
            else:
                units.append(lambda tb=tb, k=k, qq=qq, lb=lb: (
                    O.hpaged_attention(qq, pool, desc, tb, lb, H, cur_kv=k),
                    O.hpaged_append(pool, desc, tb, k, lb - 1, new_fmt)))
    case.history = None
    what = (f"the {H} kv heads of the single row" if by_head else f"the first {rows} of {w.batch} rows")
    return units, ws, step_bytes(ws, lens), what


def measure_oracle(w, budget_s, n_threads=None):
    """The oracle as it stands (plain C, fp64) on the host cores: one step of a
    bounded sample of the workload (oracle_units) with one host thread per
    unit, repeated for about budget_s seconds (median step time), and the same
    units run one after another on one thread (single_core)."""
    import concurrent.futures
    n = n_threads or host_threads()
    units, ws, nbytes, what = oracle_units(w, n)
    t_serial = 0.0
    for u in units:                       # single core: every unit once, in turn
        t = time.perf_counter()
        u()
        t_serial += time.perf_counter() - t
    walls = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(units)) as ex:
        t_all = time.perf_counter()
        while True:
            t = time.perf_counter()
            for f in [ex.submit(u) for u in units]:
                f.result()
            walls.append(time.perf_counter() - t)
            if time.perf_counter() - t_all > budget_s or len(walls) >= 200:
                break
    sec = statistics.median(walls)
    kind = "chunked" if w.chunk > 1 else "decode"
    return {"value": round(nbytes / sec / 1e9, 4), "unit": "GB/s", "cores": len(units), "kind": "oracle",
            "sample": f"{len(walls)} oracle {kind} steps (append + attention, fp64) on {what} of {w.name}, "
                      f"{len(units)} host threads (one per {'kv head' if w.batch == 1 else 'row'}); "
                      f"median {sec * 1e3:.1f} ms/step",
            "us_per_step": round(sec * 1e6, 1), "rows_tok_per_s": round(ws.batch * w.chunk / sec, 2),
            "single_core": {"value": round(nbytes / t_serial / 1e9, 4), "cores": 1,
                            "us_per_step": round(t_serial * 1e6, 1)}}


def run_reference(args, world):
    """The reference arm: the oracle, as it stands, on the host cores, for the
    headline workload (or --workload): W untimed steps, then K timed steps, each
    one step of the bounded sample with one host thread per unit."""
    import concurrent.futures
    w = workload_of(args.workload or HEADLINE)
    K = args.steps if args.steps is not None else 3
    units, ws, nbytes, what = oracle_units(w, host_threads())
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(units)) as ex:
        def step():
            for f in [ex.submit(u) for u in units]:
                f.result()
        for _ in range(args.warmup):
            step()
        t = time.perf_counter()
        for _ in range(K):
            step()
        sec = (time.perf_counter() - t) / K
    value = round(nbytes / sec / 1e9, 4)
    kind = "chunked" if w.chunk > 1 else "decode"
    cb = {"value": value, "unit": "GB/s", "cores": len(units), "kind": "oracle",
          "sample": f"{K} timed oracle {kind} steps (append + attention, fp64) on {what} of {w.name}, "
                    f"{len(units)} host threads (one per {'kv head' if w.batch == 1 else 'row'}); "
                    f"{sec * 1e3:.1f} ms/step",
          "us_per_step": round(sec * 1e6, 1), "rows_tok_per_s": round(ws.batch * w.chunk / sec, 2)}
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "layout": w.layout, "batch": w.batch, "q_heads": w.q_heads,
                       "kv_heads": w.kv_heads, "head_dim": w.head_dim, "capacity": w.capacity},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


PHASES = ("entry", "wait", "inputs", "first_tile", "warp0_tiles", "all_tiles", "cta_merged", "cluster", "end")


def phase_report(w, dev, raw_out=None):
    """Run one CUDA graph of consecutive steps with the timing build (libol_phase.so)
    and reduce its per-CTA phase stamps (%globaltimer ns and clock64 cycles at:
    entry, after the dependency wait, q and the new token loaded, first tile
    landed, warp 0's tiles done, every warp's tiles done, CTA merge done (before
    the cluster barrier), after the cluster barrier, y stored). Times are medians
    over the steps after the first: `since_prev_end` is relative to the moment the
    previous step's last CTA stored y; `per_cta` are medians over CTAs of the
    intervals between consecutive phases, from clock64."""
    import ctypes
    import torch
    import place_kv_cache_gb300 as ol
    L = ol.load(variant="phase")
    fn = L.ol_debug_phase_stamps
    fn.restype, fn.argtypes = ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32]
    s = Setup(w, dev)
    stream = torch.cuda.Stream(device=dev)
    unit = s.replicas * s.chain
    n = min(64, -(-max(unit, 32) // unit) * unit)
    with torch.cuda.stream(stream):
        for i in range(3 * unit):
            s.step(i)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                s.step(i)
        g.replay()
        stream.synchronize()
    assert fn(None, 0, 1) == 0
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    buf = np.zeros((64, 256, len(PHASES), 2), np.uint64)
    assert fn(buf.ctypes.data, buf.nbytes, 0) == 0
    if raw_out:
        np.save(raw_out, buf)
    st = buf.astype(np.int64)
    steps = [k for k in range(n) if (st[k, :, 0, 0] > 0).any()]
    ctas = [c for c in range(256) if st[steps[0], c, 0, 0] > 0]
    sub = st[:, ctas]                                     # [launch, cta, phase, 2]
    ns, cyc = sub[..., 0], sub[..., 1]
    done = ns[:, :, -1] > 0                               # CTAs that stored (mapped ones)
    # SM clock from the CTAs' own (clock64, globaltimer) spans
    span_ns = ns[steps, :, -1] - ns[steps, :, 0]
    span_cy = cyc[steps, :, -1] - cyc[steps, :, 0]
    ok = (span_ns > 0) & done[steps]
    mhz = float(np.median(span_cy[ok] / span_ns[ok] * 1e3))
    gt = np.diff(np.sort(np.unique(ns[steps][ns[steps] > 0])))
    rel = {ph: [] for ph in ("entry_first", "entry_last", "wait_first", "wait_last", "end_first", "end_last")}
    period, per_cta = [], {f"{a}->{b}": [] for a, b in zip(PHASES[1:-1], PHASES[2:])}
    for k0, k in zip(steps[:-1], steps[1:]):
        prev_end = ns[k0, done[k0], -1].max()
        m = done[k]
        period.append(ns[k, m, -1].max() - prev_end)
        for name, ph, f in (("entry", 0, None), ("wait", 1, None), ("end", -1, None)):
            rel[name + "_first"].append(ns[k, m, ph].min() - prev_end)
            rel[name + "_last"].append(ns[k, m, ph].max() - prev_end)
        for i, key in enumerate(per_cta):
            a, b = cyc[k, m, i + 1], cyc[k, m, i + 2]
            if (a > 0).all() and (b > 0).all():           # phases a plan without clusters skips stay empty
                per_cta[key].append(float(np.median(b - a)) / mhz * 1e3)
    med = lambda v: round(float(np.median(v)), 1)
    return {"workload": w.name, "phase_stamps": {
        "steps": len(steps), "ctas_per_step": len(ctas), "sm_mhz_from_clock64": round(mhz, 1),
        "globaltimer_min_step_ns": int(gt[gt > 0].min()) if (gt > 0).any() else None,
        "step_period_ns": med(period),
        "since_prev_end_ns": {k: med(v) for k, v in rel.items()},
        "per_cta_ns": {k: med(v) for k, v in per_cta.items() if v}}}


ORACLE_BUDGET_S = 4.0   # seconds of oracle steps per workload (after its one-thread pass)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world)), flush=True)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    import torch
    dev = f"cuda:{int(os.environ.get('LOCAL_RANK', 0))}"
    torch.cuda.set_device(dev)
    if args.phase_stamps:
        if rank == 0:
            print(json.dumps(phase_report(workload_of(args.workload or HEADLINE, args.rows), dev, args.phase_out)),
                  flush=True)
        return
    import place_kv_cache_gb300 as ol
    ol.load()
    head = workload_of(args.workload or HEADLINE, args.rows)
    r = measure(head, args, rank, world, dist, dev, args.steps)
    result = {"metric": METRIC, "value": r["value"], "unit": "GB/s", "n_gpus": world, "steps": r["steps"],
              "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
              "scaling": "weak", "vs_baseline": None, "dtype": r["dtype"], "data": "synthetic"}
    for k in ("us_per_step", "us_per_step_spread", "rows_tok_per_s", "pct_of_hbm_roofline", "config", "roofline",
              "gpu_launches", "device_status", "clocks"):
        result[k] = r[k]
    if "e2e" in r:
        result["e2e"] = r["e2e"]
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = measure_oracle(head, ORACLE_BUDGET_S)
    if args.workload is None:
        per = {}
        for name in PER_CONFIG:
            w = workload_of(name, args.rows)
            # a chained workload is timed over its whole chain at least
            K = None if args.steps is None else (max(args.steps, w.steps) if w.steps > 1 else args.steps)
            rr = measure(w, args, rank, world, dist, dev, K)
            if rank == 0 and not args.no_cpu_baseline:
                rr["cpu_baseline"] = measure_oracle(w, ORACLE_BUDGET_S)
            per[name] = compact(rr)
        result["per_config"] = per
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result, separators=(",", ":")), flush=True)


if __name__ == "__main__":
    main()
