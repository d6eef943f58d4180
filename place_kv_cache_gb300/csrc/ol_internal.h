// ol_internal.h -- parameter blocks passed from the host-side ABI layer
// (ol_api.cpp) to the kernel launchers (*.cu). Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime_api.h>

#include "../../include/ol.h"

namespace ol {

// Workspace layout (all offsets in bytes from the workspace base):
//   [0, 256)                     int32 device status word (+ padding)
//   [256, 256 + counters)        uint32 ticket counter per (row, kv head)
//   [partials_off, ...)          float partial results, one slot per CTA and query head:
//                                {m (log2 domain), l, o[head_dim]}
constexpr size_t kStatusBytes = 256;
constexpr int kInlineRows = 160;  // batches up to this size carry their lengths in the launch
constexpr int kMaxExtraSplits = 4096;  // CTAs beyond one per (row, kv head)

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// nq: query tokens per row (1 for a decode step, the chunk length for a
// chunked step); every query token has its own counters and partial slots.
inline size_t counters_bytes(int batch, int kv_heads, int nq = 1) {
  return align_up(sizeof(uint32_t) * (size_t)nq * (size_t)batch * (size_t)kv_heads, 256);
}
inline size_t partials_offset(int batch, int kv_heads, int nq = 1) {
  return kStatusBytes + counters_bytes(batch, kv_heads, nq);
}
inline size_t max_ctas(int batch, int kv_heads) {
  return (size_t)batch * (size_t)kv_heads + kMaxExtraSplits;
}
// A partial slot holds one CTA's state columns: the query group's heads, or for
// a chunked step up to 8 (query token, head) pairs (never more than nq * group
// columns over all of a chunk's slices, and never more than 8 per slice).
inline size_t workspace_bytes(int batch, int q_heads, int kv_heads, int head_dim, int nq = 1) {
  int group = q_heads / kv_heads;
  const size_t cols = nq > 1 ? (size_t)nq * (size_t)(group > 8 ? group : 8) : (size_t)group;
  return partials_offset(batch, kv_heads, nq) +
         cols * max_ctas(batch, kv_heads) * (size_t)(head_dim + 2) * sizeof(float);
}

// One attention / decode-step launch, fully validated on the host.
struct AttnParams {
  int layout;      // ol_layout
  int dtype;       // cache dtype (OL_F32 / OL_BF16; INT4 history with bf16 q)
  int batch, q_heads, kv_heads, group, head_dim;
  int capacity;    // tokens per row: C (contiguous / INT4) or max_pages * page_size (paged)

  // contiguous cache [2, B, Hkv, C, D]
  void* cache;
  // paged pool [2, P, Hkv, S, D] and block table [B, M]
  void* pool;
  const int32_t* block_table;
  int num_pages, page_size, max_pages;
  // INT4 planes
  uint8_t* codes;
  uint16_t* scales;
  uint8_t* zps;
  int quant_mode;
  float fixed_scale;
  int fixed_zp;
  // heterogeneous pages (pool, block_table, num_pages, page_size, max_pages as for paged)
  ol_page_format* page_fmt;  // device [num_pages]
  ol_page_format new_fmt;    // formats of the pages a fused append starts

  const void* q;        // [B, Hq, D]
  const int32_t* lens;  // device [B]
  const void* new_kv;   // [2, B, Hkv, 1, D]: appended (fused step) and attended at lens-1
  int append;           // 1: write new_kv into the cache at lens[b]-1 (fused step)
  int cur_from_new;     // 1: the token at lens[b]-1 is taken from new_kv, not the cache
  float scale;          // softmax scale
  float scale_log2;     // scale * log2(e)
  int window;           // < 0: unbounded; with nq > 1 the window of the first query token
                        // widened by nq - 1 (the union of the query tokens' ranges), for the plan
  int nq;               // query tokens per row: token z attends up to position lens - nq + z
  int tq;               // query tokens per CTA slice (state columns = group * tq, at most 8 for the
                        // tensor-core kernel); a chunked step has ceil(nq / tq) slices
  int window_q;         // the caller's window, per query token (< 0: unbounded)
  void* out;            // [B, Hq, D]
  int out_dtype;

  int inline_lens;      // 1: lengths are lens_inline (the host array, by value), lens is not read
  int early;            // 1: history rows are stable: tiles may be requested before the dependency wait
  int inputs_ready;     // 1: q and new_kv are complete at launch (host data, or written by copies
                        // ordered before the launch), so they may be read before the dependency wait
  int32_t lens_inline[kInlineRows];
  int ordered;          // 1: row_order holds the launch order of the rows (inline lengths only)
  int16_t row_order[kInlineRows];  // CTAs are assigned to rows in this order (longest work first)

  int32_t* status;      // device status word
  uint32_t* counters;   // [B * Hkv]
  float* partials;      // [max_ctas][G][D + 2]

  // split plan (host computes it from lens_host; kernels recompute the mapping from lens)
  int chunk;            // target tokens per split, a multiple of 16
  int cluster;          // CTAs per thread-block cluster (1 = no cluster)
  int variant;          // tensor-core kernel variant (warps x stages)
  int total_ctas;
  int streamk;          // 1: the CTAs split the concatenated tiles of all (row, kv head) evenly
};

// Append-only launches (CacheUpdate, PagedCacheUpdate, INT4 append).
struct AppendParams {
  int layout;
  int dtype;
  int batch, kv_heads, head_dim, capacity, new_len;
  void* cache;
  void* pool;
  const int32_t* block_table;
  int num_pages, page_size, max_pages;
  uint8_t* codes;
  uint16_t* scales;
  uint8_t* zps;
  int quant_mode;
  float fixed_scale;
  int fixed_zp;
  const void* values;        // [2, B, Hkv, new_len, D]
  const int32_t* positions;  // device [B], or NULL: every row uses scalar_position
  int scalar_position;
  int positions_are_lens;    // 1: positions[b] is a length and the append starts at positions[b] - new_len
  ol_page_format* page_fmt;  // heterogeneous pages: device [num_pages]
  ol_page_format new_fmt;    // formats of the pages the append starts
};

// Selected-page conversion of a heterogeneous paged cache.
struct QuantizeParams {
  uint8_t* pool;
  ol_page_format* page_fmt;  // device [num_pages]
  int num_pages, kv_heads, page_size, head_dim;
  const int32_t* pages;      // device [n]
  const int32_t* valid;      // device [n]
  int n;
  ol_page_format to;
};
// Visible range and split plan of one row, shared by the host planner and the
// kernels. The tokens [start, hi) (start = lo rounded down to 16) form
// ntiles 16-token tiles; they are cut into nsplit splits, split s taking tiles
// [s * ntiles / nsplit, (s + 1) * ntiles / nsplit), so splits differ by at most
// one tile. nsplit = ceil(tokens / chunk), rounded up to a multiple of
// `cluster` so that a cluster never straddles two (row, kv head).
struct RowSplit {
  int lo, hi, start, ntiles, nsplit;
};
#if defined(__CUDACC__)
__host__ __device__
#endif
inline RowSplit row_split(int n, int window, int chunk, int cluster = 1) {
  RowSplit r;
  if (n <= 0) {
    r.lo = r.hi = r.start = r.ntiles = 0;
    r.nsplit = cluster;
    return r;
  }
  r.hi = n;
  r.lo = window < 0 ? 0 : ((n - 1 - window) > 0 ? (n - 1 - window) : 0);
  r.start = r.lo & ~15;
  const int len = r.hi - r.start;
  r.ntiles = (len + 15) / 16;
  int ns = (len + chunk - 1) / chunk;
  r.nsplit = (ns + cluster - 1) / cluster * cluster;
  return r;
}

// First tile of split s (s in [0, nsplit]).
#if defined(__CUDACC__)
__host__ __device__
#endif
inline int split_tile(int s, int ntiles, int nsplit) {
  return (int)(((long long)s * ntiles) / nsplit);
}

// Element formats of the heterogeneous paged cache (host and device).
#if defined(__CUDACC__)
#define OL_HD __host__ __device__
#else
#define OL_HD
#endif
OL_HD inline int fmt_bits(int f) {
  return f == OL_FMT_F32 ? 32 : (f == OL_FMT_F16 || f == OL_FMT_BF16) ? 16
                                : (f == OL_FMT_I8 || f == OL_FMT_U8)  ? 8
                                : (f == OL_FMT_I4 || f == OL_FMT_U4)  ? 4
                                                                      : 2;
}
OL_HD inline bool fmt_affine(int f) { return f >= OL_FMT_I8 && f <= OL_FMT_U2; }
OL_HD inline bool fmt_signed(int f) { return f == OL_FMT_I8 || f == OL_FMT_I4 || f == OL_FMT_I2; }
OL_HD inline int fmt_qmin(int f) { return fmt_signed(f) ? -(1 << (fmt_bits(f) - 1)) : 0; }
OL_HD inline int fmt_qmax(int f) { return fmt_signed(f) ? (1 << (fmt_bits(f) - 1)) - 1 : (1 << fmt_bits(f)) - 1; }
// bytes of one row of D elements (D a multiple of 4)
OL_HD inline size_t fmt_row_bytes(int f, int D) { return (size_t)D * fmt_bits(f) / 8; }
#undef OL_HD

}  // namespace ol
