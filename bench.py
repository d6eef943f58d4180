"""Decode-step benchmark: achieved HBM GB/s (and % of the measured HBM
roofline), microseconds per step and rows x tokens / s of the fused decode
step (in-place append + GQA decode attention) over a caller-owned KV cache.

One step = one ``ol_decode_step`` over the whole batch of the workload: host
validation, the append of one token per row and attention over every row's
valid prefix, in one kernel launch. Steps are replayed from CUDA graphs so
the host never limits a microsecond-scale step; when one step's cache fits in
L2, consecutive steps rotate over enough independent cache replicas that the
data of a step is never L2-resident from the previous visit.

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
    ap.add_argument("--workload", default="qwen_b1_gqa7", choices=[k for k in WORKLOADS if k != "tiny_f32"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seconds", type=float, default=1.0, help="target timed seconds when --steps is not given")
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


def kernel_sources_sha() -> str:
    """sha256 over the library's device-code sources (.cu, .cuh, .h, .inc: file name
    and content, in name order): a recorded DRAM traffic figure holds only for
    the kernel sources it was measured on."""
    import hashlib
    d = os.path.join(ROOT, "place_kv_cache_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh", ".h", ".inc")):
            h.update(name.encode() + b"\0")
            with open(os.path.join(d, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes (read + write) per launch of the workload's kernel from one ncu
    capture, as listed in profiles/dram_traffic.txt; None when none was recorded
    or it was recorded on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_sources_sha()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 4 and not line.startswith("#") and parts[0] == workload and parts[3] == sha:
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
    if T > 1:
        hist = float(np.sum(lens - T)) * w.kv_heads * 2 * D * elt
        new = w.batch * w.kv_heads * T * 2 * D * elt
        return hist + 2 * new + 2 * w.batch * w.q_heads * T * D * 2   # new K/V written and read; q and y
    if w.layout == "hpaged":
        # each history token in its page's formats (K and V rows of D * bits / 8
        # bytes), plus a block-table entry and a 24-byte format pair per page
        S, M = w.page_size, w.max_pages_per_row
        cls = page_format_classes(lens, S, M)
        row = [D * (FORMAT_BITS[k[0]] + FORMAT_BITS[v[0]]) // 8 for _, (k, v) in AGE_FORMATS]
        hist = 0.0
        for b, n in enumerate(lens):
            h = int(n) - 1
            for j in range((h + S - 1) // S):
                hist += min(S, h - j * S) * row[cls[b, j]]
        hist = hist * w.kv_heads + float(np.sum(np.ceil(lens / S))) * (4 + 24)
        cur = w.batch * w.kv_heads * 2 * D * 2
        written = w.batch * w.kv_heads * row[0]
        q = w.batch * w.q_heads * D * 2
        return hist + cur + written + q + q
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
            hist = int(self.lens[b]) - 1
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


def workload_of(args):
    """The named workload, or its first --rows rows (pages sized to those rows)."""
    from workloads import scaled
    w = WORKLOADS[args.workload]
    if args.rows is not None and args.rows < w.batch:
        w = scaled(w, batch=args.rows)
        if w.layout in ("paged", "hpaged"):
            w = scaled(w, num_pages=args.rows * w.max_pages_per_row)
    return w


def run_ours(args, rank, world, dist):
    import torch
    dev = f"cuda:{int(os.environ.get('LOCAL_RANK', 0))}"
    torch.cuda.set_device(dev)
    import place_kv_cache_gb300 as ol
    ol.load()
    w = workload_of(args)
    s = Setup(w, dev, seed_offset=rank)
    stream = torch.cuda.Stream(device=dev)
    R = s.replicas
    per_graph = max(R * s.chain, 32)
    per_graph = (per_graph + R * s.chain - 1) // (R * s.chain) * (R * s.chain)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3) * R * s.chain):
            s.step(i)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(per_graph):
                s.step(i)
        g.replay()
        stream.synchronize()
    # calibrate the step time to size the timed region
    t = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(5):
            g.replay()
    stream.synchronize()
    est = (time.perf_counter() - t) / (5 * per_graph)
    if args.steps is None:
        K = max(per_graph, int(args.seconds / max(est, 1e-7)) // per_graph * per_graph)
    else:
        K = max(per_graph, (args.steps + per_graph - 1) // per_graph * per_graph)
    n_graphs = K // per_graph
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(int(os.environ.get("LOCAL_RANK", 0))) as clk:
        with torch.cuda.stream(stream):
            for _ in range(max(1, int(0.3 / max(est * per_graph, 1e-6)))):
                g.replay()                       # keep the GPU busy while the sampler settles
        if dist is not None:
            dist.barrier()
        stream.synchronize()
        clk.mark_start()
        # one event between consecutive graphs (recorded on the same stream, no
        # synchronization between them): per-graph step times for the spread
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(n_graphs - 1)]
        with torch.cuda.stream(stream):
            e0.record(stream)
            for k in range(n_graphs):
                g.replay()
                if k < n_graphs - 1:
                    marks[k].record(stream)
            e1.record(stream)
        stream.synchronize()
        clk.mark_end()
        if dist is not None:
            dist.barrier()
    ms = e0.elapsed_time(e1)
    bounds = [e0] + marks + [e1]
    per_graph_us = sorted(bounds[k].elapsed_time(bounds[k + 1]) * 1e3 / per_graph for k in range(n_graphs))
    spread = {"graphs": n_graphs,
              "p10": round(float(np.percentile(per_graph_us, 10)), 3),
              "median": round(float(np.percentile(per_graph_us, 50)), 3),
              "p90": round(float(np.percentile(per_graph_us, 90)), 3)}
    ms_per_step, gbs = combine_ranks(ms, K, s.bytes_per_step, world, dist, device=dev)
    status = ol.ol_workspace_status(s.ws, stream=stream)
    peak, peak_src = measured_peaks()
    result = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"int4": "u4+bf16", "hpaged": "bf16+i8+i4/u4 pages, f32 math"}.get(w.layout, "bf16"), "data": "synthetic",
        "us_per_step": round(ms_per_step * 1e3, 3),
        "us_per_step_spread": dict(spread, note=f"per graph of {per_graph} steps, rank {rank}"),
        "rows_tok_per_s": round(w.batch * world / (ms_per_step * 1e-3), 1),
        "pct_of_hbm_roofline": round(100.0 * gbs / world / peak, 2),
        "config": {"workload": w.name, "layout": w.layout, "batch": w.batch, "q_heads": w.q_heads,
                   "kv_heads": w.kv_heads, "head_dim": w.head_dim, "capacity": w.capacity,
                   "lens_mean": float(np.mean(s.lens)), "bytes_per_step": s.bytes_per_step,
                   "l2": s.l2_note, "graph_steps": per_graph, "chained_steps": s.chain,
                   "history_stable": s.chain == 1,
                   "parallelism": f"rows x{world} (independent)"},
        "roofline": {"bound": "hbm", "achieved": round(gbs / world, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / world / peak, 4), "traffic": recorded_traffic(w.name),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else
                     "fallback 6.8 TB/s"},
        "gpu_launches": K,
        "device_status": status,
        "clocks": clk.summary(),
    }
    if not args.no_e2e and w.chunk == 1 and w.layout != "hpaged":
        result["e2e"] = run_e2e(s, stream, K_e2e=min(K, 200 * R))
    elif not args.no_e2e:
        # the host-buffer call serves the decode step of the uniform layouts; chunked
        # steps and heterogeneous pages run from device buffers
        result["e2e"] = None
    if w.chunk > 1:
        result["config"]["chunk"] = w.chunk
    return result


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
            "call": "ol_decode_step_host (one C-ABI call per step, pinned host buffers)",
            "transfer": "q, new K/V loaded and y stored by the step's kernels from/to mapped pinned host memory"}


# --------------------------------------------------------------- oracle

def oracle_step_inputs(w, max_rows):
    """A bounded sample of the workload for the CPU oracle: the first max_rows rows."""
    import oracle as O
    from workloads import scaled
    rows = min(w.batch, max_rows)
    ws = scaled(w, batch=rows)
    if w.layout == "hpaged":   # the sample's rows own their pages; a pool of the full size is not needed
        ws = scaled(ws, num_pages=rows * w.max_pages_per_row)
    case = make_case(ws, seed=w.seed, history_len_offset=w.chunk)
    return O, ws, case


def run_oracle_steps(w, budget_s, max_rows):
    """Time the oracle's decode step (append + attention) on a sample of the workload."""
    from workloads import block_table, contiguous_cache, poisoned_pool
    O, ws, case = oracle_step_inputs(w, max_rows)
    if w.layout == "contiguous" and w.chunk > 1:
        cache = contiguous_cache(case)
        T = w.chunk
        rng = np.random.default_rng(w.seed + 7)
        q = bf16_from_f32(rng.standard_normal((ws.batch, ws.q_heads, T, ws.head_dim)).astype(np.float32))
        kv = bf16_from_f32(rng.standard_normal((2, ws.batch, ws.kv_heads, T, ws.head_dim)).astype(np.float32))

        def one():
            O.cache_update(cache, kv, case.lens - T)
            return O.chunk_attention(q, cache, case.lens, T)
    elif w.layout == "contiguous":
        cache = contiguous_cache(case)

        def one():
            O.cache_update(cache, case.new_kv, case.lens - 1)
            return O.decode_attention(case.q, cache, case.lens)
    elif w.layout == "paged":
        pool = poisoned_pool(ws)
        table = block_table(case)
        for b, h in enumerate(case.history):
            if h.shape[2]:
                O.paged_update(pool, table[b:b + 1], h[:, None], [0])

        def one():
            O.paged_update(pool, table, case.new_kv, case.lens - 1)
            return O.paged_attention(case.q, pool, table, case.lens)
    elif w.layout == "hpaged":
        S, M, H, D = ws.page_size, ws.max_pages_per_row, ws.kv_heads, ws.head_dim
        pool, desc = O.hpaged_pool(ws.num_pages, H, S, D)
        table = block_table(case)
        cls = page_format_classes(case.lens, S, M)
        for b, h in enumerate(case.history):
            for j in range((h.shape[2] + S - 1) // S):
                k, v = AGE_FORMATS[cls[b, j]][1]
                O.hpaged_append(pool, desc, table[b:b + 1], h[:, None, :, j * S:(j + 1) * S], [j * S],
                                O.page_desc(k=k, v=v))
        new_fmt = O.page_desc(*AGE_FORMATS[0][1])

        def one():
            y = O.hpaged_attention(case.q, pool, desc, table, case.lens, H, cur_kv=case.new_kv)
            O.hpaged_append(pool, desc, table, case.new_kv, case.lens - 1, new_fmt)
            return y
    else:
        planes = O.int4_planes(ws.batch, ws.kv_heads, ws.capacity, ws.head_dim)
        for b, h in enumerate(case.history):
            sub = O.int4_planes(1, ws.kv_heads, ws.capacity, ws.head_dim)
            O.int4_append(*sub, h[:, None], [0])
            for full, part in zip(planes, sub):
                full[:, b] = part[:, 0]

        def one():
            O.int4_append(*planes, case.new_kv, case.lens - 1)
            return O.int4_attention(case.q, *planes, case.lens, cur_kv=case.new_kv)
    times = []
    t_all = time.perf_counter()
    while True:
        t = time.perf_counter()
        one()
        times.append(time.perf_counter() - t)
        if time.perf_counter() - t_all > budget_s or len(times) >= 1000:
            break
    sec = statistics.median(times)
    nbytes = step_bytes(ws, case.lens)
    return {"value": round(nbytes / sec / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{len(times)} oracle {'chunked' if w.chunk > 1 else 'decode'} steps (append + attention, "
                      f"fp64) on the first {ws.batch} of "
                      f"{w.batch} rows of {w.name}; median {sec * 1e3:.1f} ms/step",
            "us_per_step": round(sec * 1e6, 1), "rows_tok_per_s": round(ws.batch / sec, 2)}


def run_reference(args, rank, world):
    w = WORKLOADS[args.workload]
    max_rows = {"qwen_b1_gqa7": 1, "ragged_b32": 4, "paged_b64": 2, "int4_b16": 1, "chunk4_b32": 1,
                "hpaged_b64": 2}[w.name]
    K = args.steps if args.steps is not None else 3
    budget = 60.0
    res = run_oracle_steps(w, budget_s=min(budget, 10.0 * max(1, K)), max_rows=max_rows)
    return {"impl": "reference", "metric": METRIC, "value": res["value"], "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": res["us_per_step"] / 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "layout": w.layout, "batch": w.batch, "q_heads": w.q_heads,
                       "kv_heads": w.kv_heads, "head_dim": w.head_dim, "capacity": w.capacity},
            "cpu_baseline": res,
            "e2e": {"value": res["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    result = run_ours(args, rank, world, dist)
    if rank == 0 and not args.no_cpu_baseline:
        w = WORKLOADS[args.workload]
        max_rows = {"qwen_b1_gqa7": 1, "ragged_b32": 4, "paged_b64": 2, "int4_b16": 1, "chunk4_b32": 1,
                "hpaged_b64": 2}[w.name]
        result["cpu_baseline"] = run_oracle_steps(w, budget_s=10.0, max_rows=max_rows)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


if __name__ == "__main__":
    main()
