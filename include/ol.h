/*
 * ol.h -- C ABI of the GB300 decode step over a caller-owned KV cache.
 *
 * One operation, in three cache layouts: append this step's K/V in place
 * ("CacheUpdate": page "Mutable execution cache", sections Value model,
 * Required alias, Model example and Runtime contract) fused with single-token
 * attention softmax(q K^T * scale) V over the valid prefix (page "Persistent
 * input/output feedback", section Optional heterogeneous paged KV: causal
 * masking, left_window_size, grouped-query attention, online softmax, current
 * K/V attended before they are encoded).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers are DEVICE pointers unless the name ends in `_host`. The caller
 *   owns every buffer: caches, q, values, outputs, block tables, workspace.
 *   The library keeps no pointer after a call returns, apart from the
 *   (base, size, owner) triples of ol_cache_bind.
 * - The library allocates nothing: no cudaMalloc, no output cache, no copy
 *   fallback. The only memory it touches is what the caller passes.
 * - Every call validates everything on the host before any launch. A non-OK
 *   return means nothing was written and nothing was launched. OL_OK means
 *   the work was enqueued on `stream` (asynchronous with respect to the host).
 * - Required alias: `updated_*` must equal the descriptor's data pointer on
 *   every call (pointer identity), else OL_ERR_ALIAS. The descriptor must be
 *   OL_READ_WRITE, else OL_ERR_READONLY. Capacity is part of the shape:
 *   position + new_len > capacity is OL_ERR_CAPACITY, never growth.
 * - Lengths: lens[b] counts the tokens row b attends, including the token this
 *   step appends; the append position of a decode step is lens[b] - 1.
 *   `*_host` arrays drive validation and launch sizing; `*_dev` arrays (same
 *   values, on the device) drive the kernels. The caller keeps them equal;
 *   the kernels still check every index they use and skip (never perform) an
 *   access outside the caller's buffers, recording OL_DEVICE_GUARD in the
 *   workspace status word where a workspace is passed. For attention and
 *   step calls on batches of at most 160 rows the launch carries lens_host by
 *   value and the kernels read no lens_dev; a call captured in a CUDA graph
 *   replays the lengths (and launch size) it was captured with.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream). Calls on one workspace must not overlap on the GPU.
 * - Alignment: every device pointer must be 16-byte aligned (OL_ERR_ALIGN).
 * - dtype: OL_BF16 (bit pattern of bfloat16) or OL_F32. q and new K/V share
 *   the cache's dtype; the attention output is OL_BF16 or OL_F32.
 */
#ifndef OL_H_
#define OL_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define OL_API __attribute__((visibility("default")))
#else
#define OL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef void* ol_stream; /* cudaStream_t */

typedef enum ol_status {
  OL_OK = 0,
  OL_ERR_NULL = 1,         /* a required pointer is NULL */
  OL_ERR_ALIAS = 2,        /* updated pointer != cache pointer, or an input/output overlaps the cache */
  OL_ERR_READONLY = 3,     /* descriptor access is OL_READ_ONLY but the call writes the cache */
  OL_ERR_CAPACITY = 4,     /* position + new_len > capacity, or lens[b] outside [0, capacity] */
  OL_ERR_SHAPE = 5,        /* inconsistent sizes (q_heads not a multiple of kv_heads, ...) */
  OL_ERR_DTYPE = 6,        /* unknown dtype, or a dtype the layout does not take */
  OL_ERR_BUSY = 7,         /* the cache range is bound by another owner (ol_cache_bind) */
  OL_ERR_WORKSPACE = 8,    /* workspace NULL or smaller than ol_workspace_size() */
  OL_ERR_CUDA = 9,         /* a CUDA runtime call failed (launch error, bad stream, ...) */
  OL_ERR_UNSUPPORTED = 10, /* a valid request this build does not implement */
  OL_ERR_INJECTED = 11,    /* host fault injection: env OL_FAULT_INJECT=after_validate */
  OL_ERR_PAGE = 12,        /* a block-table entry is outside the pool, or two rows append to one slot */
  OL_ERR_ALIGN = 13        /* a device pointer is not 16-byte aligned */
} ol_status;

typedef enum ol_dtype { OL_F32 = 0, OL_BF16 = 1 } ol_dtype;

/* ValueInfoProto.access of the cache binding (page "Mutable execution cache", Proto additions). */
typedef enum ol_access { OL_READ_ONLY = 0, OL_READ_WRITE = 1 } ol_access;

/*
 * Optional bit ORed into a descriptor's `access`: the caller guarantees that
 * no work enqueued earlier on the same stream is still writing this cache's
 * history rows [0, lens[b] - 1) of any row (nor, for a paged cache, the block
 * table entries that cover them). Attention-bearing calls may then start
 * reading those rows while the preceding kernel finishes (programmatic
 * dependent launch); q, new K/V, lengths, outputs and workspace are still
 * touched only after it completes. Typical use: consecutive layers of a model,
 * each with its own cache. Not valid for a step that immediately follows a
 * step on the same cache (that step wrote row lens[b] - 2).
 */
enum { OL_HISTORY_STABLE = 0x100 };

typedef enum ol_layout {
  OL_LAYOUT_CONTIGUOUS = 0,
  OL_LAYOUT_PAGED = 1,
  OL_LAYOUT_INT4 = 2,
  OL_LAYOUT_HPAGED = 3 /* ol_hpaged_kv: paged, every page with its own K and V formats */
} ol_layout;

/* How an INT4 append chooses (scale, zero point) per block of 32 values. */
typedef enum ol_quant_mode {
  OL_Q_DYNAMIC = 0, /* lo = min(0, min x), hi = max(0, max x), scale = fp16((hi-lo)/15) (1 if 0),
                       zp = sat(round_half_even(-lo/scale)) */
  OL_Q_FIXED = 1    /* scale = fp16(fixed_scale), zp = fixed_zp for every block */
} ol_quant_mode;

/*
 * Launch tuning. The library plans every launch itself (kernel variant, split
 * length, cluster size, CTA waves) from the call's sizes and the device. For
 * measurement and for test coverage of the plans it does not pick by default,
 * the environment variable OL_TUNE, read once per process at the first call
 * that plans a launch, overrides parts of the plan: a comma-separated list of
 * key=value with keys waves (CTA waves of a split plan), minchunk (smallest
 * split, tokens), cfg (tensor-core variant 0..4), cluster (largest cluster
 * size), cpu (clusters per row and kv head), generic (1: CUDA-core kernel for
 * heterogeneous pages), hpwaves and cwaves (CTA waves of heterogeneous-page and
 * chunked plans). Unknown keys and out-of-range values are ignored. Results
 * stay within the same tolerances under every setting; only speed changes.
 */

/* Device status word values (ol_workspace_status). */
enum { OL_DEVICE_OK = 0, OL_DEVICE_GUARD = 1 };

/*
 * Contiguous cache [2, batch, kv_heads, capacity, head_dim], K plane 0,
 * V plane 1, row-major, dtype OL_BF16 or OL_F32. Capacity is in the shape
 * (page "Mutable execution cache", Model example: cache
 * FLOAT16[2, batch, heads, max_length, head_size]).
 * `owner` identifies the session for ol_cache_bind (0 = none).
 */
typedef struct ol_kv_cache {
  void* data;
  int32_t dtype;
  int32_t batch, kv_heads, capacity, head_dim;
  int32_t access;
  uint64_t owner;
} ol_kv_cache;

/*
 * Paged cache: one fixed pool [2, num_pages, kv_heads, page_size, head_dim]
 * (K plane 0, V plane 1) and a block table [batch, max_pages] of int32 page
 * indices: logical token t of row b lives in slot t % page_size of page
 * block_table[b][t / page_size] (page "Mutable execution cache", ONNX Runtime
 * GenAI: logical pages map to slices of the num_blocks axis of a pool that
 * never grows). The capacity of a row is max_pages * page_size.
 * `block_table_host` is the same table in host memory, used for validation.
 */
typedef struct ol_paged_kv {
  void* data;
  const int32_t* block_table;
  const int32_t* block_table_host;
  int32_t dtype;
  int32_t num_pages, kv_heads, page_size, head_dim;
  int32_t batch, max_pages;
  int32_t access;
  uint64_t owner;
} ol_paged_kv;

/*
 * INT4 blockwise-affine cache, stored as three planes of the logical
 * [2, batch, kv_heads, capacity, head_dim] cache (head_dim a multiple of 64):
 *   codes  uint8 [2, batch, kv_heads, capacity, head_dim / 2]   two uint4 codes per byte, low nibble first
 *   scales fp16  [2, batch, kv_heads, capacity, head_dim / 32]  one scale per block of 32 values
 *   zps    uint8 [2, batch, kv_heads, capacity, head_dim / 64]  two uint4 zero points per byte, low first
 * Reconstruction: (code - zp) * scale (page "Custom quantized and persistent
 * values", Struct types and byte-encodable layouts: blocked affine, packing
 * least-significant bits first). `codes` is the alias pointer.
 */
typedef struct ol_int4_kv {
  uint8_t* codes;
  uint16_t* scales;
  uint8_t* zps;
  int32_t batch, kv_heads, capacity, head_dim;
  int32_t quant_mode;
  float fixed_scale;
  int32_t fixed_zp;
  int32_t access;
  uint64_t owner;
} ol_int4_kv;

/*
 * Heterogeneous paged cache: every page stores its K and its V in its own
 * format (page "Persistent input/output feedback", sections Optional
 * heterogeneous paged KV and Selected-block quantization). Formats: dense
 * FLOAT, FLOAT16, BFLOAT16; affine INT8, UINT8, INT4, UINT4, INT2, UINT2 with
 * value = (code - zero_point) * scale, one scalar (scale, zero point) per page
 * and plane. Encoding is QuantizeLinear in IEEE fp32:
 * code = saturate(round_half_even(x / scale) + zero_point); dense formats
 * round to nearest even. Codes of four and two bits pack two and four per
 * byte, least-significant bits first (page "Custom, quantized, and persistent
 * values", affine branch).
 */
typedef enum ol_page_format_id {
  OL_FMT_F32 = 0, OL_FMT_F16 = 1, OL_FMT_BF16 = 2,
  OL_FMT_I8 = 3, OL_FMT_U8 = 4, OL_FMT_I4 = 5, OL_FMT_U4 = 6, OL_FMT_I2 = 7, OL_FMT_U2 = 8
} ol_page_format_id;

/* One plane's format; scale and zero_point are ignored by dense formats. Affine
   formats need a positive finite scale and a zero point inside the code range. */
typedef struct ol_plane_format {
  int32_t format;
  float scale;
  int32_t zero_point;
} ol_plane_format;

typedef struct ol_page_format {
  ol_plane_format k, v;
} ol_page_format;

/*
 * The heterogeneous pool: num_pages slots of 2 * kv_heads * page_size *
 * head_dim * 4 bytes (room for the widest format). Plane k (0 = K, 1 = V) of
 * page p starts at byte p * slot + k * slot / 2; in a plane of format f the
 * codes of (head h, page slot s) start at (h * page_size + s) * row_bytes(f)
 * and hold head_dim elements (row_bytes = head_dim * bits / 8). head_dim must
 * be a multiple of 4. Logical token t of row b lives in slot t % page_size of
 * page block_table[b][t / page_size].
 *   formats       device [num_pages]: each page's formats, read by the kernels
 *   formats_host  host [num_pages]: the same table, read by the host to
 *                 validate and plan. Calls that start or convert a page update
 *                 both: the host entry when the call is made, the device entry
 *                 in stream order.
 * `pool` is the alias pointer.
 */
typedef struct ol_hpaged_kv {
  void* pool;
  ol_page_format* formats;
  ol_page_format* formats_host;
  const int32_t* block_table;
  const int32_t* block_table_host;
  int32_t num_pages, kv_heads, page_size, head_dim;
  int32_t batch, max_pages;
  int32_t access;
  uint64_t owner;
} ol_hpaged_kv;

/* Human-readable name of a status code (static string). */
OL_API const char* ol_status_string(ol_status s);

/* ABI version of this header (major * 100 + minor). */
OL_API int32_t ol_version(void);

/*
 * Bytes of workspace the attention and step calls need for these sizes. The
 * workspace holds the split-K partial results, one ticket counter per
 * (row, kv head) and the device status word. Zero it once with
 * ol_workspace_init before its first use; each call leaves its counters at
 * zero when it completes.
 */
OL_API size_t ol_workspace_size(int32_t batch, int32_t q_heads, int32_t kv_heads, int32_t head_dim);

/* Zero a workspace on `stream` (cudaMemsetAsync of the caller's memory). */
OL_API ol_status ol_workspace_init(void* workspace, size_t ws_bytes, ol_stream stream);

/*
 * Read and clear the workspace's device status word (synchronizes `stream`).
 * *status_out is OL_DEVICE_OK, or OL_DEVICE_GUARD if a kernel skipped an
 * access because a device-side index disagreed with the validated sizes.
 */
OL_API ol_status ol_workspace_status(void* workspace, int32_t* status_out, ol_stream stream);

/*
 * Bind a writable cache range [base, base + bytes) to `owner` (page "Mutable
 * execution cache", Runtime contract: one writable cache binding cannot be
 * used concurrently by multiple sessions). Binding a range that overlaps a
 * range bound by another owner returns OL_ERR_BUSY; rebinding one's own range
 * is OL_OK. While bound, calls whose descriptor overlaps the range with a
 * different `owner` return OL_ERR_BUSY. Unbinding a range one does not own
 * returns OL_ERR_BUSY; unbinding an unbound range is OL_OK.
 */
OL_API ol_status ol_cache_bind(const void* base, size_t bytes, uint64_t owner);
OL_API ol_status ol_cache_unbind(const void* base, uint64_t owner);

/*
 * CacheUpdate(cache, values, position) -> updated_cache, with updated_cache
 * aliasing cache (page "Mutable execution cache", Value model and Model
 * example). values [2, batch, kv_heads, new_len, head_dim] is written to rows
 * [position, position + new_len) of every (plane, row, head); nothing else is
 * written. position is the INT64 scalar of the page's example.
 * Errors: NULL, ALIAS, READONLY, CAPACITY (position < 0 or
 * position + new_len > capacity), SHAPE, DTYPE, BUSY, ALIGN, CUDA.
 */
OL_API ol_status ol_cache_update(const ol_kv_cache* cache, void* updated_cache, const void* values,
                          int32_t new_len, int64_t position, ol_stream stream);

/* As ol_cache_update with one position per row (positions_host/dev [batch] int32). */
OL_API ol_status ol_cache_update_rows(const ol_kv_cache* cache, void* updated_cache, const void* values,
                               int32_t new_len, const int32_t* positions_host,
                               const int32_t* positions_dev, ol_stream stream);

/*
 * PagedCacheUpdate(cache, page_id, values, position): write values
 * [2, batch, kv_heads, new_len, head_dim] to logical tokens
 * [p_b, p_b + new_len) of each row through the block table, in place
 * (page "Mutable execution cache", Heterogeneous paged cache and Runtime
 * contract: existing pages are updated in place, nothing is allocated).
 * Every page the write reaches must be in [0, num_pages) and no two rows
 * may write the same slot (OL_ERR_PAGE).
 */
OL_API ol_status ol_paged_cache_update(const ol_paged_kv* kv, void* updated_pool, const void* values,
                                int32_t new_len, const int32_t* positions_host,
                                const int32_t* positions_dev, ol_stream stream);

/*
 * Decode attention over a contiguous cache (read-only use of the cache): the
 * Attention contract of page "Persistent input/output feedback", sections
 * Optional heterogeneous paged KV and Versioned operator schema (causal by
 * default, left_window_size, query heads a multiple of the KV heads, online
 * softmax over the valid and visible tokens only, Y in the dtype of Q unless
 * fp32 is asked for) over the cache layout of page "Mutable execution cache",
 * section Model example.
 * q [batch, q_heads, head_dim] (cache dtype); out [batch, q_heads, head_dim]
 * in out_dtype. Query head h reads kv head h / (q_heads / kv_heads). Row b
 * attends its visible tokens: [0, lens[b]) if window < 0, else
 * [max(0, lens[b] - 1 - window), lens[b]). lens[b] == 0 gives out = 0.
 * scale <= 0 selects 1/sqrt(head_dim).
 * Errors: NULL, ALIAS (q, out, lens_dev or workspace overlapping the cache;
 * out overlapping q or the workspace), CAPACITY (lens[b] outside
 * [0, capacity]), SHAPE, DTYPE, WORKSPACE, BUSY, ALIGN, UNSUPPORTED
 * (head_dim > 256), CUDA.
 */
OL_API ol_status ol_decode_attention(const ol_kv_cache* cache, const void* q, int32_t q_heads,
                              const int32_t* lens_host, const int32_t* lens_dev, float scale,
                              int32_t window, void* out, int32_t out_dtype, void* workspace,
                              size_t ws_bytes, ol_stream stream);

/*
 * Decode attention over a paged cache: the same Attention contract (page
 * "Persistent input/output feedback", section Optional heterogeneous paged
 * KV) over a fixed pool addressed through the block table (page "Mutable
 * execution cache", section ONNX Runtime GenAI: logical pages map to slices of
 * the pool). Arguments, visibility and errors as ol_decode_attention; every
 * page the visible range reaches must be in [0, num_pages) (OL_ERR_PAGE).
 */
OL_API ol_status ol_paged_decode_attention(const ol_paged_kv* kv, const void* q, int32_t q_heads,
                                    const int32_t* lens_host, const int32_t* lens_dev,
                                    float scale, int32_t window, void* out, int32_t out_dtype,
                                    void* workspace, size_t ws_bytes, ol_stream stream);

/*
 * INT4 append: quantize values_bf16 [2, batch, kv_heads, 1, head_dim] per
 * block of 32 (round half to even, saturate to [0, 15]; page "Persistent
 * input/output feedback", quantization paragraph) and write codes, scales and
 * zero points at row positions[b] of each (plane, row, head). updated_codes
 * must equal cache->codes.
 */
OL_API ol_status ol_int4kv_append(const ol_int4_kv* cache, void* updated_codes, const void* values_bf16,
                           const int32_t* positions_host, const int32_t* positions_dev,
                           ol_stream stream);

/*
 * INT4 decode attention. History is reconstructed from the codes. If cur_kv
 * ([2, batch, kv_heads, 1, head_dim] bf16) is non-NULL, the token at
 * lens[b] - 1 takes part uncompressed from cur_kv instead of the codes (the
 * current K/V are attended before they are encoded: page "Persistent
 * input/output feedback", section Optional heterogeneous paged KV).
 * q is bf16; otherwise as ol_decode_attention.
 */
OL_API ol_status ol_int4kv_decode_attention(const ol_int4_kv* cache, const void* q, int32_t q_heads,
                                     const int32_t* lens_host, const int32_t* lens_dev,
                                     const void* cur_kv, float scale, int32_t window, void* out,
                                     int32_t out_dtype, void* workspace, size_t ws_bytes,
                                     ol_stream stream);

/*
 * The fused decode step in one launch: append new_kv
 * [2, batch, kv_heads, 1, head_dim] at position lens[b] - 1 of every row
 * (CacheUpdate / PagedCacheUpdate / INT4 append, in place, `updated` aliasing
 * the descriptor's data pointer) and attend [visible range of lens[b]] with
 * the new token included. For OL_LAYOUT_INT4 the new token is attended
 * uncompressed and stored encoded. `cache_desc` points to the ol_kv_cache,
 * ol_paged_kv or ol_int4_kv that `layout` names. new_kv has the cache dtype
 * (bf16 for INT4). Requires lens[b] >= 1.
 */
OL_API ol_status ol_decode_step(int32_t layout, const void* cache_desc, void* updated, const void* q,
                         int32_t q_heads, const void* new_kv, const int32_t* lens_host,
                         const int32_t* lens_dev, float scale, int32_t window, void* out,
                         int32_t out_dtype, void* workspace, size_t ws_bytes, ol_stream stream);

/*
 * Append new_len tokens per row to a heterogeneous paged cache: values
 * [2, batch, kv_heads, new_len, head_dim] bf16 at positions[b].. of every row.
 * A token that lands in slot 0 of its page starts that page: the page takes
 * the formats *new_pages (the caller's format selection for this call, chosen
 * from anything it likes, e.g. the retained length); every other token is
 * encoded in its page's existing formats, so earlier pages are never converted
 * and a partially filled page keeps its format. `updated` must equal
 * cache->pool. Writes only the appended slots and the started pages' formats.
 */
OL_API ol_status ol_hpaged_append(const ol_hpaged_kv* cache, void* updated, const void* values_bf16,
                                  int32_t new_len, const int32_t* positions_host, const int32_t* positions_dev,
                                  const ol_page_format* new_pages, ol_stream stream);

/*
 * Decode attention over a heterogeneous paged cache: every visible token is
 * decoded with its page's formats. If cur_kv ([2, batch, kv_heads, 1,
 * head_dim] bf16) is non-NULL the token at lens[b] - 1 takes part
 * uncompressed from cur_kv (current K/V attended before they are encoded).
 * q bf16 [batch, q_heads, head_dim]; otherwise as ol_decode_attention.
 */
OL_API ol_status ol_hpaged_decode_attention(const ol_hpaged_kv* cache, const void* q, int32_t q_heads,
                                            const int32_t* lens_host, const int32_t* lens_dev, const void* cur_kv,
                                            float scale, int32_t window, void* out, int32_t out_dtype,
                                            void* workspace, size_t ws_bytes, ol_stream stream);

/*
 * The fused step on a heterogeneous paged cache: append new_kv
 * [2, batch, kv_heads, 1, head_dim] bf16 at lens[b] - 1 (as ol_hpaged_append,
 * pages started by it taking *new_pages) and attend with the new token
 * uncompressed, in one launch.
 */
OL_API ol_status ol_hpaged_decode_step(const ol_hpaged_kv* cache, void* updated, const void* q, int32_t q_heads,
                                       const void* new_kv, const ol_page_format* new_pages,
                                       const int32_t* lens_host, const int32_t* lens_dev, float scale,
                                       int32_t window, void* out, int32_t out_dtype, void* workspace,
                                       size_t ws_bytes, ol_stream stream);

/*
 * Chunked step on a heterogeneous paged cache (as ol_chunk_step): query token
 * i of row b at lens[b] - new_len + i attends its causal, windowed range; the
 * chunk's tokens take part uncompressed from new_kv [2, batch, kv_heads,
 * new_len, head_dim] bf16 and are then encoded into their pages (as
 * ol_hpaged_append at lens[b] - new_len: pages the chunk starts take
 * *new_pages). q and out [batch, q_heads, new_len, head_dim]. Two launches:
 * the attention, then the append; every check runs before the first.
 * ws_bytes >= ol_workspace_size_chunk(batch, q_heads, kv_heads, head_dim, new_len).
 */
OL_API ol_status ol_hpaged_chunk_step(const ol_hpaged_kv* cache, void* updated, const void* q, int32_t q_heads,
                                      int32_t new_len, const void* new_kv, const ol_page_format* new_pages,
                                      const int32_t* lens_host, const int32_t* lens_dev, float scale,
                                      int32_t window, void* out, int32_t out_dtype, void* workspace,
                                      size_t ws_bytes, ol_stream stream);

/*
 * QuantizePagedCache on selected pages (page "Persistent input/output
 * feedback", section Selected-block quantization): for each of the n pages
 * (unique indices), the first valid[i] slots of every head are decoded in the
 * page's current formats and encoded in *to (K and V independently; dense
 * targets dequantize), the other slots become the target format's zeros, and
 * the page's formats become *to. Unselected pages are untouched. Every index,
 * length and format is checked before anything is written. pages and valid are
 * given in host memory (validation) and device memory (the kernel), equal.
 */
OL_API ol_status ol_hpaged_quantize(const ol_hpaged_kv* cache, void* updated, const int32_t* pages_host,
                                    const int32_t* pages_dev, const int32_t* valid_host, const int32_t* valid_dev,
                                    int32_t n, const ol_page_format* to, ol_stream stream);

/*
 * Chunked step: multi-token append with causal attention inside the chunk
 * (the Attention contract of page "Persistent input/output feedback", section
 * Optional heterogeneous paged KV: causal by default, left window, every new
 * token visible to itself and to the later tokens of the chunk). For every
 * row b: write new_kv [2, batch, kv_heads, new_len, head_dim] at positions
 * lens[b] - new_len .. lens[b] - 1 (in place, `updated` aliasing the
 * descriptor's data pointer), then for every query token i of
 * q [batch, q_heads, new_len, head_dim] attend positions
 * [max(0, pos_i - window), pos_i] with pos_i = lens[b] - new_len + i
 * (window < 0: [0, pos_i]) into out [batch, q_heads, new_len, head_dim].
 * new_len = 1 is ol_decode_step. Contiguous, paged and INT4 caches (not the
 * heterogeneous pool: OL_ERR_UNSUPPORTED). INT4: the chunk's tokens take
 * part uncompressed from new_kv (bf16) and are quantized into the cache only
 * after the attention (the same section: current K/V are attended as
 * uncompressed values and encoded afterwards); history comes from the codes.
 * Requires new_len <= lens[b] <= capacity and ws_bytes >=
 * ol_workspace_size_chunk(batch, q_heads, kv_heads, head_dim, new_len).
 * Two launches on `stream` (contiguous and paged: the append, then one
 * attention launch whose grid slice z serves query token z; INT4: the
 * attention, then the append); every check runs before the first.
 */
OL_API size_t ol_workspace_size_chunk(int32_t batch, int32_t q_heads, int32_t kv_heads, int32_t head_dim,
                                      int32_t new_len);
OL_API ol_status ol_chunk_step(int32_t layout, const void* cache_desc, void* updated, const void* q,
                               int32_t q_heads, int32_t new_len, const void* new_kv, const int32_t* lens_host,
                               const int32_t* lens_dev, float scale, int32_t window, void* out, int32_t out_dtype,
                               void* workspace, size_t ws_bytes, ol_stream stream);

/*
 * Storage statistics of a call (page "Persistent input/output feedback",
 * sections Opt-in storage auditing through runtime events and Optional
 * heterogeneous paged KV: the storage_* reports and the direct call's
 * copied / dequantized byte counts). The library records them, on the
 * calling host thread, for every append, attention or decode-step call that
 * passes validation (also when the launch then fails: the counts describe the
 * work the call requested). They are host arithmetic on the call's sizes; no
 * device work is added.
 */
typedef struct {
  int64_t calls;                       /* calls summed into this record */
  int64_t storage_allocations;         /* KV storage allocations: always 0 (caches are caller-owned, never grown) */
  int64_t storage_allocated_bytes;     /* KV storage bytes requested: always 0 */
  int64_t storage_prefix_copied_bytes; /* bytes of the valid prefix copied: always 0 (appends write in place) */
  int64_t storage_append_copied_bytes; /* new payload bytes stored by appends (INT4: codes + scales + zero points) */
  int64_t storage_reuse_count;         /* K / V storage tensors appended in place (2 per appending call) */
  int64_t dequantized_bytes;           /* FLOAT bytes decoded from quantized history: 4 per element per (token,
                                          kv head, K or V), the current uncompressed token excluded; one decode
                                          serves the whole query group */
  int64_t attended_tokens;             /* sum over query tokens, rows and kv heads of the visible tokens, the
                                          current one included */
  int64_t kv_payload_bytes_read;       /* K/V payload bytes of the visible history read from the cache, summed
                                          over query tokens (a chunk's query tokens share most of it) */
  int64_t workspace_bytes;             /* workspace bytes the call's shapes require (bound on its scratch) */
} ol_stats;

/* The record of the last validated call on this thread (zeros before the first). */
OL_API ol_status ol_last_call_stats(ol_stats* out);
/* Sums of every record on this thread since the last ol_reset_stats (calls > 1). */
OL_API ol_status ol_total_stats(ol_stats* out);
OL_API void ol_reset_stats(void);

/*
 * Workspace bytes for ol_decode_step_host: those of ol_workspace_size plus
 * device staging for q, new_kv, the lengths and y (sized for 4-byte elements,
 * so one size serves every dtype). 0 on invalid sizes.
 */
OL_API size_t ol_workspace_size_host(int32_t batch, int32_t q_heads, int32_t kv_heads, int32_t head_dim);

/*
 * The fused decode step with host-resident inputs and output: q_host
 * [batch, q_heads, head_dim], new_kv_host [2, batch, kv_heads, 1, head_dim]
 * (dtypes as for ol_decode_step), lens_host [batch] and y in out_host
 * [batch, q_heads, head_dim] of out_dtype. Each of q_host, new_kv_host and
 * out_host that is page-locked host memory mapped into the device's address
 * space (cudaHostAlloc'd or pinned tensors; registered memory with mapping)
 * and 16-byte aligned is used in place: the step's kernels load from it and
 * store y into it across the CPU-GPU link, with no copy. Any other host
 * buffer goes through the workspace's staging area with host-to-device /
 * device-to-host copies on `stream` (pageable memory at the driver's pace).
 * The lengths travel in the launch for up to 160 rows, else by one copy.
 * Everything is asynchronous: out_host holds y once `stream` has been
 * synchronized, and the host buffers must stay valid and unchanged until
 * then; out_host overlapping q_host or new_kv_host is OL_ERR_ALIAS. The cache stays in
 * device memory, described as for ol_decode_step. ws_bytes must be at least
 * ol_workspace_size_host(batch, q_heads, kv_heads, head_dim).
 * Errors: those of ol_decode_step (the descriptor, host pointers, lengths and
 * workspace size are checked before any copy is enqueued; a call that fails
 * later has written only the staging area), or OL_ERR_CUDA if a copy cannot
 * be enqueued. The cache is never touched by a failing call.
 */
OL_API ol_status ol_decode_step_host(int32_t layout, const void* cache_desc, void* updated, const void* q_host,
                                     int32_t q_heads, const void* new_kv_host, const int32_t* lens_host,
                                     float scale, int32_t window, void* out_host, int32_t out_dtype,
                                     void* workspace, size_t ws_bytes, ol_stream stream);

/*
 * The fused decode step with no allocation by anyone: no workspace argument.
 * The method's pages describe no such call; it exists for callers that cannot call
 * cudaMalloc -- code running inside a host engine that owns all device memory
 * and forbids allocation while it executes (an inference-engine plugin's
 * enqueue, a fixed-arena runtime), or a latency-critical decode loop that
 * cannot afford an allocation's implicit synchronization.
 *
 * Its scratch (split-K partials, ticket counters, status word) is one
 * file-scope device array of OL_NOALLOC_SCRATCH_BYTES inside this library;
 * every GPU that loads the library holds it until the process exits. The
 * first call on a device looks up that array's device address (with the
 * device current); make that first call before any stream capture. Every
 * check of ol_decode_step runs first, with the array as the workspace: a
 * request whose worst-case workspace, ol_workspace_size(batch, q_heads,
 * kv_heads, head_dim), exceeds OL_NOALLOC_SCRATCH_BYTES is OL_ERR_WORKSPACE,
 * and any rejected call returns ol_decode_step's status for the same
 * arguments with nothing enqueued. A call that passes clears the array's
 * counters and status word on `stream` (cudaMemsetAsync of the array itself,
 * no allocation) and then runs ol_decode_step with the array as its
 * workspace. All calls share the one array: calls that overlap on the GPU (on
 * different streams, or from different threads) race on it and must not be
 * issued. The heterogeneous-page layout is not taken (as by ol_decode_step,
 * which has no format choice for the pages it would start).
 */
#define OL_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
OL_API ol_status ol_decode_step_noalloc(int32_t layout, const void* cache_desc, void* updated, const void* q,
                                        int32_t q_heads, const void* new_kv, const int32_t* lens_host,
                                        const int32_t* lens_dev, float scale, int32_t window, void* out,
                                        int32_t out_dtype, ol_stream stream);

/*
 * Read and clear the device status word of the current device's
 * allocation-free scratch (synchronizes `stream`): OL_DEVICE_OK, or
 * OL_DEVICE_GUARD if a kernel of an ol_decode_step_noalloc call skipped an
 * access because a device-side index disagreed with the validated sizes (as
 * ol_workspace_status for a caller's workspace). Every ol_decode_step_noalloc
 * call clears the word before it runs, so the word reports the calls since the
 * last one that started, i.e. the most recent call.
 */
OL_API ol_status ol_noalloc_status(int32_t* status_out, ol_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* OL_H_ */
