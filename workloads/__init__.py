"""Seeded synthetic inputs for the decode step over a caller-owned KV cache.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests. It holds none of the method's arithmetic: it only draws random
numbers in a fixed order, rounds them to the storage type, and describes the
workload shapes. Anything that places tokens into a cache layout (the append,
the page table lookup, INT4 quantization) lives on either side of the boundary
— the oracle or the kernels — never here.

Draw order for one case, from one ``numpy.random.default_rng(seed)``:
lengths -> page permutation -> q -> per row b: K history, V history ->
new K -> new V.

bf16 values are produced from float32 draws by round-to-nearest-even on the
bit pattern. Spare cache capacity is filled with the bf16 quiet NaN 0x7FC0 (or
float32 NaN) as poison, so any read outside the valid range shows up as NaN.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

BF16_NAN = np.uint16(0x7FC0)
F32_NAN = np.float32(np.nan)


def bf16_from_f32(a) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bit patterns."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = a.view(np.uint32)
    # u + 0x7FFF + (bit 16 of u), shifted down 16: in uint32 this cannot wrap
    # for any non-NaN pattern (at most 0xFF800000 + 0x8000); NaNs are replaced below
    r = u >> np.uint32(16)
    r &= np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    out = r.astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def bf16_to_f32(u) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    u = np.ascontiguousarray(np.asarray(u, dtype=np.uint16))
    return (u.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape of one decode-step workload.

    ``lens`` semantics: the number of attended tokens of row b, including the
    token appended by this step; the append position is ``lens[b] - 1``.
    """
    name: str
    dtype: str                 # "f32" or "bf16"
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    capacity: int              # tokens per row (contiguous / INT4) or pages*page_size (paged)
    layout: str                # "contiguous" | "paged" | "int4" | "hpaged" (per-page formats)
    seed: int
    lens_fixed: Optional[int] = None          # every row has this length
    lens_range: Optional[tuple] = None        # inclusive uniform range, drawn per row
    page_size: int = 0
    num_pages: int = 0
    steps: int = 1                             # chained decode steps
    dist: str = "normal"                       # "normal" (N(0,1)) or "uniform" (U[-1,1])
    block: int = 32                            # INT4 block along head_dim
    chunk: int = 1                             # tokens appended and attended per row per step

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def max_pages_per_row(self) -> int:
        return self.capacity // self.page_size if self.page_size else 0


# The five synthetic workloads of the decode step (page: "Mutable execution
# cache" §Model example for the contiguous cache shape; "Persistent
# input/output feedback" §Optional heterogeneous paged KV for page size 16 and
# INT4 formats).
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", "f32", 1, 1, 1, 4, 16, "contiguous", seed=0,
                         lens_fixed=1, steps=4, dist="uniform"),
    "qwen_b1_gqa7": Workload("qwen_b1_gqa7", "bf16", 1, 28, 4, 128, 8192, "contiguous",
                             seed=2, lens_fixed=4097),
    "ragged_b32": Workload("ragged_b32", "bf16", 32, 32, 8, 128, 8192, "contiguous",
                           seed=3, lens_range=(512, 8192)),
    "paged_b64": Workload("paged_b64", "bf16", 64, 32, 8, 128, 16384, "paged", seed=4,
                          lens_range=(1, 16384), page_size=16, num_pages=65536),
    "int4_b16": Workload("int4_b16", "bf16", 16, 32, 8, 128, 32768, "int4", seed=5,
                         lens_fixed=16385, steps=64),
    # chunked step (multi-token append, causal inside the chunk): the ragged
    # shape with 4 tokens per row per step, as a speculative-decoding verifier
    # appends and scores its drafted tokens
    "chunk4_b32": Workload("chunk4_b32", "bf16", 32, 32, 8, 128, 8192, "contiguous",
                           seed=6, lens_range=(512, 8192), chunk=4),
    # the INT4 cache of int4_b16 taking 4 tokens per row per step (chunked step:
    # the chunk attended uncompressed, then quantized into the cache)
    "int4chunk4_b16": Workload("int4chunk4_b16", "bf16", 16, 32, 8, 128, 32768, "int4", seed=8,
                               lens_fixed=16388, chunk=4),
    # heterogeneous pages: the paged shape with every page's K/V formats chosen
    # by its age (AGE_FORMATS): recent pages BFLOAT16, older INT8, oldest 4-bit
    "hpaged_b64": Workload("hpaged_b64", "bf16", 64, 32, 8, 128, 16384, "hpaged", seed=7,
                           lens_range=(1, 16384), page_size=16, num_pages=65536),
    # the heterogeneous pages taking 4 tokens per row per step (chunked step:
    # the chunk attended uncompressed, then encoded into its pages)
    "hpchunk4_b64": Workload("hpchunk4_b64", "bf16", 64, 32, 8, 128, 16384, "hpaged", seed=9,
                             lens_range=(8, 16384), page_size=16, num_pages=65536, chunk=4),
}

# Page formats of the heterogeneous workloads, as (format, scale, zero point)
# for K and for V; format codes FLOAT 0, FLOAT16 1, BFLOAT16 2, INT8 3, UINT8 4,
# INT4 5, UINT4 6, INT2 7, UINT2 8. The formats are a caller's policy (page
# "Persistent input/output feedback", §Optional heterogeneous paged KV: the
# caller picks each page's format, for example from the retained length): a
# page whose last slot is fewer than `age` tokens behind the row's end takes
# the first entry that admits it. Scales fit N(0, 1) values: INT8 at 1/32
# covers +/-3.97, INT4 and UINT4 (zero point 8) at 0.5 cover -4..3.5.
AGE_FORMATS = ((1024, ((2, 1.0, 0), (2, 1.0, 0))),
               (4096, ((3, 0.03125, 0), (3, 0.03125, 0))),
               (None, ((5, 0.5, 0), (6, 0.5, 8))))


def page_format_classes(lens: np.ndarray, page_size: int, max_pages: int, ages=AGE_FORMATS) -> np.ndarray:
    """[B, max_pages] index into ``ages`` of each logical page's format (pages
    past a row's end get the class of age 0, the format a new page starts in)."""
    out = np.zeros((len(lens), max_pages), np.int32)
    for b, n in enumerate(lens):
        for j in range(max_pages):
            age = max(int(n) - (j + 1) * page_size, 0)
            out[b, j] = next(i for i, (lim, _) in enumerate(ages) if lim is None or age < lim)
    return out


def _draw(rng: np.random.Generator, shape, dist: str) -> np.ndarray:
    if dist == "normal":
        return rng.standard_normal(size=shape, dtype=np.float32)
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, size=shape).astype(np.float32)
    raise ValueError(dist)


def _store(a: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_from_f32(a) if dtype == "bf16" else np.ascontiguousarray(a, dtype=np.float32)


def _poison(shape, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return np.full(shape, BF16_NAN, dtype=np.uint16)
    return np.full(shape, F32_NAN, dtype=np.float32)


def draw_lens(rng: np.random.Generator, w: Workload) -> np.ndarray:
    if w.lens_fixed is not None:
        return np.full(w.batch, w.lens_fixed, dtype=np.int32)
    lo, hi = w.lens_range
    return rng.integers(lo, hi + 1, size=w.batch, dtype=np.int64).astype(np.int32)


@dataclasses.dataclass
class Case:
    """One seeded decode-step input set.

    q        [B, Hq, D]            query of the token being decoded
    lens     [B] int32             attended tokens per row, including the new one
    history  list over b of [2, Hkv, lens[b]-1, D]  (K plane 0, V plane 1)
    new_kv   [2, B, Hkv, 1, D]     K/V of the token appended at lens[b]-1
    perm     page permutation (paged layout only), else None
    Values are uint16 bf16 bit patterns or float32, per ``dtype``.
    """
    workload: Workload
    lens: np.ndarray
    q: np.ndarray
    history: list
    new_kv: np.ndarray
    perm: Optional[np.ndarray]

    @property
    def dtype(self) -> str:
        return self.workload.dtype


def make_case(w: Workload, *, lens: Optional[np.ndarray] = None, seed: Optional[int] = None,
              history_len_offset: int = 1) -> Case:
    """Draw one case. ``history_len_offset`` tokens of each row are left for the
    append (1 for a decode step); use 0 to get a history of ``lens[b]`` tokens."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    if lens is None:
        lens = draw_lens(rng, w)       # explicit lengths skip this draw
    else:
        lens = np.asarray(lens, dtype=np.int32)
    perm = None
    if w.layout in ("paged", "hpaged"):
        perm = rng.permutation(w.num_pages).astype(np.int32)
    D = w.head_dim
    q = _store(_draw(rng, (w.batch, w.q_heads, D), w.dist), w.dtype)
    history = []
    for b in range(w.batch):
        h = max(int(lens[b]) - history_len_offset, 0)
        k = _store(_draw(rng, (w.kv_heads, h, D), w.dist), w.dtype)
        v = _store(_draw(rng, (w.kv_heads, h, D), w.dist), w.dtype)
        history.append(np.stack([k, v]))
    nk = _store(_draw(rng, (w.batch, w.kv_heads, 1, D), w.dist), w.dtype)
    nv = _store(_draw(rng, (w.batch, w.kv_heads, 1, D), w.dist), w.dtype)
    return Case(w, lens, q, history, np.stack([nk, nv]), perm)


def contiguous_cache(case: Case, capacity: Optional[int] = None) -> np.ndarray:
    """Lay the drawn history into a fresh [2, B, Hkv, C, D] cache whose spare
    capacity is NaN poison. Token t of row b lives at index t of that row:
    this is the contiguous layout itself, written out."""
    w = case.workload
    C = w.capacity if capacity is None else capacity
    cache = _poison((2, w.batch, w.kv_heads, C, w.head_dim), case.dtype)
    for b, h in enumerate(case.history):
        n = h.shape[2]
        cache[:, b, :, :n, :] = h
    return cache


def block_table(case: Case) -> np.ndarray:
    """Row b's logical pages map to perm[b*M : (b+1)*M] (M = max pages per row)."""
    w = case.workload
    M = w.max_pages_per_row
    return np.ascontiguousarray(case.perm[: w.batch * M].reshape(w.batch, M))


def poisoned_pool(w: Workload) -> np.ndarray:
    """A fresh paged pool [2, num_pages, Hkv, page_size, D] filled with NaN poison."""
    return _poison((2, w.num_pages, w.kv_heads, w.page_size, w.head_dim), w.dtype)


def scaled(w: Workload, **changes) -> Workload:
    """The same workload with some fields replaced (used for reduced-size parity cases)."""
    return dataclasses.replace(w, **changes)


def fixture_signed_ramp(batch: int, heads: int, length: int, head_dim: int, step: float,
                        coef: float = 0.173) -> np.ndarray:
    """Components +/-(coef*step) with sign (-1)^(d+h): the four-step fixture values
    (page "Persistent input/output feedback", §Optional heterogeneous paged KV,
    tolerance table). Returns float32 [batch, heads, length, head_dim]."""
    d = np.arange(head_dim)
    h = np.arange(heads)
    sign = np.where(((d[None, :] + h[:, None]) % 2) == 0, 1.0, -1.0).astype(np.float32)
    a = np.float32(coef * step) * sign
    return np.ascontiguousarray(np.broadcast_to(a[None, :, None, :], (batch, heads, length, head_dim)),
                                dtype=np.float32)
