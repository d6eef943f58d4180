// ol_api.cpp -- the C ABI declared in include/ol.h: host-side validation,
// the cache bind registry, the split-K launch plan and kernel dispatch.
//
// Every check runs before any launch, so an error return means nothing was
// written (page "Mutable execution cache", Runtime contract: overflow is an
// error, never growth; read-only initializers are never mutable caches; one
// writable binding is not used concurrently by several sessions; Required
// alias: pointer identity checked, no silent copy fallback).
#include <cmath>
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "ol_internal.h"
#include "ol_launch.h"

namespace ol {
namespace {

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
  bool empty() const { return hi <= lo; }
};
Range range_of(const void* p, size_t bytes) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return {a, a + bytes};
}
bool overlaps(Range a, Range b) { return !a.empty() && !b.empty() && a.lo < b.hi && b.lo < a.hi; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Binding {
  uintptr_t lo, hi;
  uint64_t owner;
};
std::mutex g_bind_mu;
std::vector<Binding> g_bindings;

ol_status check_owner(const Range* ranges, int nranges, uint64_t owner) {
  std::lock_guard<std::mutex> lk(g_bind_mu);
  for (const Binding& bd : g_bindings)
    for (int i = 0; i < nranges; ++i)
      if (overlaps(ranges[i], Range{bd.lo, bd.hi}) && bd.owner != owner) return OL_ERR_BUSY;
  return OL_OK;
}

bool fault_injected() {
  const char* v = std::getenv("OL_FAULT_INJECT");
  return v && std::strcmp(v, "after_validate") == 0;
}

size_t elt_bytes(int dtype) { return dtype == OL_F32 ? 4 : 2; }
bool valid_dtype(int d) { return d == OL_F32 || d == OL_BF16; }

// Launch tuning: OL_TUNE="waves=<w>,minchunk=<c>,cfg=<variant>,cluster=<cs>,cpu=<k>,generic=<0|1>,hpwaves=<w>,
// cwaves=<w>" (read once).
struct Tune {
  int waves = -1;  // CTA waves of a split plan without clusters; -1 = by layout (measured best)
  int min_chunk = 16;
  int cfg = -1;      // tensor-core kernel variant; -1 = default
  int cluster = -1;  // cluster size cap; -1 = automatic
  int clusters_per_unit = -1;  // cap on clusters per (row, kv head) for small batches
  bool generic = false;        // heterogeneous pages: the CUDA-core kernel even where the tensor-core one applies
  int hp_waves = 1;            // heterogeneous pages: CTA waves of the split plan (hpaged_b64, rows
                               // longest-first: 1 wave 287.5 us/step, 2 299.1, 3 310.3, 4 308.3)
  int chunk_waves = 1;         // chunked steps on tensor cores (measured best on chunk4_b32)
};
const Tune& tune() {
  static Tune t = [] {
    Tune x;
    const char* v = std::getenv("OL_TUNE");
    if (!v) return x;
    std::string s(v);
    size_t pos = 0;
    while (pos < s.size()) {
      size_t comma = s.find(',', pos);
      std::string kv = s.substr(pos, comma == std::string::npos ? std::string::npos : comma - pos);
      size_t eq = kv.find('=');
      if (eq != std::string::npos) {
        std::string k = kv.substr(0, eq);
        int val = std::atoi(kv.c_str() + eq + 1);
        if (k == "waves" && val > 0) x.waves = val;
        if (k == "minchunk" && val >= 16) x.min_chunk = (val + 15) / 16 * 16;
        if (k == "cfg" && val >= 0 && val <= 4) x.cfg = val;
        if (k == "cluster" && val >= 1) x.cluster = val;
        if (k == "cpu" && val >= 1) x.clusters_per_unit = val;
        if (k == "generic") x.generic = val != 0;
        if (k == "hpwaves" && val > 0) x.hp_waves = val;
        if (k == "cwaves" && val > 0) x.chunk_waves = val;
      }
      if (comma == std::string::npos) break;
      pos = comma + 1;
    }
    return x;
  }();
  return t;
}

int pow2_floor(long long x) {
  int r = 1;
  while ((long long)r * 2 <= x) r *= 2;
  return r;
}

// Pick the target split length so that about `target` CTAs cover all
// (row, kv head) visible token ranges, within the workspace's CTA budget.
void plan_splits(AttnParams& p, const int32_t* lens_host, long long target, int cluster) {
  long long tok = 0;
  for (int b = 0; b < p.batch; ++b) {
    RowSplit rs = row_split(lens_host[b], p.window, 16);
    tok += rs.hi - rs.start;
  }
  tok *= p.kv_heads;
  long long chunk = target > 0 ? (tok + target - 1) / target : tok;
  chunk = (chunk + 15) / 16 * 16;
  if (chunk < tune().min_chunk) chunk = tune().min_chunk;
  const long long budget = (long long)max_ctas(p.batch, p.kv_heads);
  for (;;) {
    long long total = 0;
    for (int b = 0; b < p.batch; ++b) total += row_split(lens_host[b], p.window, (int)chunk, cluster).nsplit;
    total *= p.kv_heads;
    if (total <= budget || chunk >= (1ll << 30)) {
      p.chunk = (int)chunk;
      p.cluster = cluster;
      p.total_ctas = (int)total;
      return;
    }
    chunk *= 2;
  }
}

// Tensor-core paths: kernel variant (warps x stages), CTAs per SM, and for
// batches with fewer (row, kv head) units than SMs one wave of CTAs grouped in
// clusters that merge their splits through distributed shared memory.
void plan_fast(AttnParams& p, const int32_t* lens_host, int sms, int force_variant = -1) {
  const long long units = (long long)p.batch * p.kv_heads;
  const bool int4 = p.layout == OL_LAYOUT_INT4;
  // measured defaults: 8 warps x 2 stages for contiguous caches and small
  // batches, 4 warps x 2 stages (three CTAs per SM) for paged pools; INT4:
  // 6 warps x 6 stages (chunked steps 8 x 4)
  if (force_variant >= 0)
    p.variant = force_variant;
  else if (tune().cfg >= 0)
    p.variant = tune().cfg;
  else if (int4)
    p.variant = 0;
  else
    p.variant = (units >= sms && p.layout == OL_LAYOUT_PAGED) ? 2 : 3;
  if (int4 && p.variant > 2) p.variant = 0;
  if (!int4 && p.nq > 1 && p.variant != 2) p.variant = 3;  // chunked steps: the variants built for them
  const int smem = (int4 ? fast_int4_smem(p.variant) : fast_bf16_smem(p.variant)) + 1024;
  const int warps = int4 ? fast_int4_warps(p.variant) : fast_bf16_warps(p.variant);
  int per_sm = (228 * 1024) / smem;
  if (per_sm > 64 / warps) per_sm = 64 / warps;
  // INT4: the CTAs per SM its launch bounds promise (registers and shared memory)
  if (int4) per_sm = fast_int4_ctas_per_sm(p.variant, p.nq > 1);
  if (per_sm < 1) per_sm = 1;
  const long long slots = (long long)sms * per_sm;
  p.streamk = 0;
  if (int4 && units > 0 && slots <= 4096 && tune().cluster <= 0) {
    // Stream-K: the INT4 kernel is bound by instruction throughput, so every
    // SM gets the same number of tiles (whole CTAs per (row, kv head) leave
    // some SMs with more). Used when every row has tiles and a CTA gets at
    // least 64 of them (its extra segment costs little against that).
    long long tiles = 0;
    bool empty_row = false;
    for (int b = 0; b < p.batch; ++b) {
      const int nt = row_split(lens_host[b], p.window, 16).ntiles;
      empty_row |= nt == 0;
      tiles += nt;
    }
    tiles *= p.kv_heads;
    if (!empty_row && tiles >= 64 * slots) {
      p.streamk = 1;
      p.cluster = 1;
      p.chunk = 16;
      p.total_ctas = (int)slots;
      return;
    }
  }
  if (units >= sms || units == 0) {
    // CTA waves, measured with the rows launched longest-first: contiguous
    // caches 1 (ragged_b32: 79.5 us/step; 2 waves 84.1, 3 87.5), paged pools 2
    // (paged_b64: 345.4; 3 waves 345.4, 4 346.8, 6 350.7), INT4 2
    const int waves = tune().waves > 0 ? tune().waves
                                       : (p.layout == OL_LAYOUT_CONTIGUOUS ? 1 : 2);
    plan_splits(p, lens_host, slots * (p.nq > 1 ? tune().chunk_waves : waves), 1);
    return;
  }
  int cs = pow2_floor(slots / units);
  if (cs > 16) cs = 16;
  const int cap = int4 ? fast_int4_max_cluster(p.variant) : fast_bf16_max_cluster(p.variant, p.layout == OL_LAYOUT_PAGED);
  if (cs > cap) cs = cap;
  if (tune().cluster > 0 && cs > tune().cluster) cs = pow2_floor(tune().cluster);
  // one cluster per (row, kv head) by default: a second level of merging
  // through global memory costs more than the extra CTAs gain
  long long k = slots / (units * cs);
  const long long kcap = tune().clusters_per_unit > 0 ? tune().clusters_per_unit : 1;
  if (k > kcap) k = kcap;
  if (k < 1) k = 1;
  int longest = 0;
  for (int b = 0; b < p.batch; ++b) {
    RowSplit rs = row_split(lens_host[b], p.window, 16);
    if (rs.hi - rs.start > longest) longest = rs.hi - rs.start;
  }
  long long chunk = (longest + cs * k - 1) / (cs * k);
  chunk = (chunk + 15) / 16 * 16;
  if (chunk < 16) chunk = 16;
  long long total = 0;
  for (int b = 0; b < p.batch; ++b) total += row_split(lens_host[b], p.window, (int)chunk, cs).nsplit;
  p.chunk = (int)chunk;
  p.cluster = cs;
  p.total_ctas = (int)(total * p.kv_heads);
  // Consecutive decode steps overlap (each requests its first tiles while the
  // previous one runs) only when both steps' clusters are resident together.
  // The 8-warp variant holds one CTA per SM; when it cannot hold two steps'
  // clusters, the 6-warp variant (two CTAs per SM) does. Measured at
  // B = 1, 7 query heads per kv head, 4097 tokens: 6.16 -> 5.72 us/step at
  // 4 kv heads, 7.25 -> 6.44 at 7; at 1-3 kv heads the 8-warp one is faster.
  if (force_variant < 0 && tune().cfg < 0 && !int4 && p.nq == 1 && p.variant == 3 && cs > 1) {
    const long long clusters = p.total_ctas / cs;
    if (2 * clusters > fast_bf16_active_clusters(3, p.layout == OL_LAYOUT_PAGED, cs))
      plan_fast(p, lens_host, sms, 4);
  }
}

// Launch order of the rows of a split plan (lengths carried by value): rows
// by descending tiles per CTA, so the longest CTAs start in the first wave and
// the short ones fill the tail (longest first). Stream-K plans balance by
// construction and keep row order.
void order_rows(AttnParams& p, const int32_t* lens_host) {
  p.ordered = 0;
  if (!p.inline_lens || p.streamk || p.batch < 2) return;
  std::vector<std::pair<int, int>> key(p.batch);  // (tiles per CTA, row)
  for (int b = 0; b < p.batch; ++b) {
    const RowSplit rs = row_split(lens_host[b], p.window, p.chunk, p.cluster);
    key[b] = {rs.nsplit > 0 ? (rs.ntiles + rs.nsplit - 1) / rs.nsplit : 0, b};
  }
  std::stable_sort(key.begin(), key.end(),
                   [](const std::pair<int, int>& x, const std::pair<int, int>& y) { return x.first > y.first; });
  for (int i = 0; i < p.batch; ++i) p.row_order[i] = (int16_t)key[i].second;
  p.ordered = 1;
}

int sm_count_cached() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// ----------------------------------------------------------- descriptors

struct CacheView {
  int layout;
  int dtype;
  int batch, kv_heads, head_dim, capacity;
  int access;
  bool history_stable;
  uint64_t owner;
  void* alias_ptr;  // pointer that `updated` must equal
  Range ranges[3];  // cache storage (INT4: three planes)
  int nranges;
};

ol_status view_contiguous(const ol_kv_cache* c, CacheView& v) {
  if (!c || !c->data) return OL_ERR_NULL;
  if (!valid_dtype(c->dtype)) return OL_ERR_DTYPE;
  if (c->batch < 0 || c->kv_heads <= 0 || c->capacity < 0 || c->head_dim <= 0) return OL_ERR_SHAPE;
  if (!aligned16(c->data)) return OL_ERR_ALIGN;
  v = {};
  v.layout = OL_LAYOUT_CONTIGUOUS;
  v.dtype = c->dtype;
  v.batch = c->batch;
  v.kv_heads = c->kv_heads;
  v.head_dim = c->head_dim;
  v.capacity = c->capacity;
  v.access = c->access & ~OL_HISTORY_STABLE;
  v.history_stable = (c->access & OL_HISTORY_STABLE) != 0;
  v.owner = c->owner;
  v.alias_ptr = c->data;
  v.ranges[0] = range_of(c->data, 2ull * c->batch * c->kv_heads * c->capacity * c->head_dim * elt_bytes(c->dtype));
  v.nranges = 1;
  return OL_OK;
}

ol_status view_paged(const ol_paged_kv* c, CacheView& v) {
  if (!c || !c->data || !c->block_table || !c->block_table_host) return OL_ERR_NULL;
  if (!valid_dtype(c->dtype)) return OL_ERR_DTYPE;
  if (c->batch < 0 || c->kv_heads <= 0 || c->num_pages <= 0 || c->page_size <= 0 || c->head_dim <= 0 ||
      c->max_pages < 0)
    return OL_ERR_SHAPE;
  if ((long long)c->max_pages * c->page_size > (1ll << 30)) return OL_ERR_SHAPE;
  if (!aligned16(c->data) || !aligned16(c->block_table)) return OL_ERR_ALIGN;
  v = {};
  v.layout = OL_LAYOUT_PAGED;
  v.dtype = c->dtype;
  v.batch = c->batch;
  v.kv_heads = c->kv_heads;
  v.head_dim = c->head_dim;
  v.capacity = c->max_pages * c->page_size;
  v.access = c->access & ~OL_HISTORY_STABLE;
  v.history_stable = (c->access & OL_HISTORY_STABLE) != 0;
  v.owner = c->owner;
  v.alias_ptr = c->data;
  v.ranges[0] = range_of(c->data, 2ull * c->num_pages * c->kv_heads * c->page_size * c->head_dim *
                                      elt_bytes(c->dtype));
  v.nranges = 1;
  return OL_OK;
}

ol_status view_int4(const ol_int4_kv* c, CacheView& v) {
  if (!c || !c->codes || !c->scales || !c->zps) return OL_ERR_NULL;
  if (c->batch < 0 || c->kv_heads <= 0 || c->capacity < 0 || c->head_dim <= 0) return OL_ERR_SHAPE;
  if (c->head_dim % 64 != 0) return OL_ERR_SHAPE;
  if (c->quant_mode != OL_Q_DYNAMIC && c->quant_mode != OL_Q_FIXED) return OL_ERR_SHAPE;
  if (c->quant_mode == OL_Q_FIXED &&
      (!(c->fixed_scale > 0.f) || !std::isfinite(c->fixed_scale) || c->fixed_zp < 0 || c->fixed_zp > 15))
    return OL_ERR_SHAPE;
  if (!aligned16(c->codes) || !aligned16(c->scales) || !aligned16(c->zps)) return OL_ERR_ALIGN;
  v = {};
  v.layout = OL_LAYOUT_INT4;
  v.dtype = OL_BF16;
  v.batch = c->batch;
  v.kv_heads = c->kv_heads;
  v.head_dim = c->head_dim;
  v.capacity = c->capacity;
  v.access = c->access & ~OL_HISTORY_STABLE;
  v.history_stable = (c->access & OL_HISTORY_STABLE) != 0;
  v.owner = c->owner;
  v.alias_ptr = c->codes;
  const unsigned long long rows = 2ull * c->batch * c->kv_heads * c->capacity;
  v.ranges[0] = range_of(c->codes, rows * (c->head_dim / 2));
  v.ranges[1] = range_of(c->scales, rows * (c->head_dim / 32) * 2);
  v.ranges[2] = range_of(c->zps, rows * (c->head_dim / 64));
  v.nranges = 3;
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (overlaps(v.ranges[i], v.ranges[j])) return OL_ERR_ALIAS;
  return OL_OK;
}

bool valid_plane_format(const ol_plane_format& f) {
  if (f.format < OL_FMT_F32 || f.format > OL_FMT_U2) return false;
  if (!fmt_affine(f.format)) return true;
  return f.scale > 0.f && std::isfinite(f.scale) && f.zero_point >= fmt_qmin(f.format) &&
         f.zero_point <= fmt_qmax(f.format);
}
bool valid_page_format(const ol_page_format& f) { return valid_plane_format(f.k) && valid_plane_format(f.v); }

// Bytes of one page slot of a heterogeneous pool: room for both planes in fp32.
size_t hpaged_slot_bytes(const ol_hpaged_kv* c) { return 2ull * c->kv_heads * c->page_size * c->head_dim * 4; }

ol_status view_hpaged(const ol_hpaged_kv* c, CacheView& v) {
  if (!c || !c->pool || !c->formats || !c->formats_host || !c->block_table || !c->block_table_host)
    return OL_ERR_NULL;
  if (c->batch < 0 || c->kv_heads <= 0 || c->num_pages <= 0 || c->page_size <= 0 || c->head_dim <= 0 ||
      c->max_pages < 0 || c->head_dim % 4 != 0)
    return OL_ERR_SHAPE;
  if ((long long)c->max_pages * c->page_size > (1ll << 30)) return OL_ERR_SHAPE;
  if (!aligned16(c->pool) || !aligned16(c->block_table) || (reinterpret_cast<uintptr_t>(c->formats) & 3u))
    return OL_ERR_ALIGN;
  v = {};
  v.layout = OL_LAYOUT_HPAGED;
  v.dtype = OL_BF16;  // q, new tokens and outputs' input side are bf16
  v.batch = c->batch;
  v.kv_heads = c->kv_heads;
  v.head_dim = c->head_dim;
  v.capacity = c->max_pages * c->page_size;
  v.access = c->access & ~OL_HISTORY_STABLE;
  v.history_stable = (c->access & OL_HISTORY_STABLE) != 0;
  v.owner = c->owner;
  v.alias_ptr = c->pool;
  v.ranges[0] = range_of(c->pool, (size_t)c->num_pages * hpaged_slot_bytes(c));
  v.ranges[1] = range_of(c->formats, sizeof(ol_page_format) * (size_t)c->num_pages);
  v.nranges = 2;
  if (overlaps(v.ranges[0], v.ranges[1])) return OL_ERR_ALIAS;
  return OL_OK;
}

// The same pool seen as a plain paged cache, for the block-table checks.
ol_paged_kv paged_shape_of(const ol_hpaged_kv* c) {
  ol_paged_kv k = {};
  k.data = c->pool;
  k.block_table = c->block_table;
  k.block_table_host = c->block_table_host;
  k.num_pages = c->num_pages;
  k.kv_heads = c->kv_heads;
  k.page_size = c->page_size;
  k.head_dim = c->head_dim;
  k.batch = c->batch;
  k.max_pages = c->max_pages;
  k.dtype = OL_BF16;
  return k;
}

// Formats in force for token t of row b during an append that starts at pos:
// the started pages' (slot 0 inside the append) new formats, else the page's.
const ol_page_format& hpaged_token_format(const ol_hpaged_kv* c, int b, int t, int pos, const ol_page_format& nf) {
  const int page = c->block_table_host[(size_t)b * c->max_pages + t / c->page_size];
  return t - t % c->page_size >= pos ? nf : c->formats_host[page];
}

// Heterogeneous page checks (after check_pages on the block table): every page
// that a call reads, or appends into without starting it, has valid formats.
// read_hi[b]: tokens [lo, read_hi) of row b are read from the cache, lo from
// the window; pos/new_len: the append (new_len 0 for none).
ol_status check_hpaged_formats(const ol_hpaged_kv* c, const int32_t* lens, int window, const int32_t* read_hi,
                               const int32_t* pos, int new_len) {
  const int S = c->page_size;
  for (int b = 0; b < c->batch; ++b) {
    if (lens) {
      const RowSplit rs = row_split(lens[b], window, 1);
      for (int t = rs.lo; t < read_hi[b]; t += S - t % S)
        if (!valid_page_format(c->formats_host[c->block_table_host[(size_t)b * c->max_pages + t / S]]))
          return OL_ERR_SHAPE;
    }
    if (new_len > 0 && pos[b] % S != 0 &&
        !valid_page_format(c->formats_host[c->block_table_host[(size_t)b * c->max_pages + pos[b] / S]]))
      return OL_ERR_SHAPE;
  }
  return OL_OK;
}

// After a validated append: the host mirror takes the started pages' formats.
void hpaged_start_pages(const ol_hpaged_kv* c, const int32_t* pos, int new_len, const ol_page_format& nf) {
  const int S = c->page_size;
  for (int b = 0; b < c->batch; ++b)
    for (int t = (pos[b] + S - 1) / S * S; t < pos[b] + new_len; t += S)
      c->formats_host[c->block_table_host[(size_t)b * c->max_pages + t / S]] = nf;
}

ol_status view_of(int layout, const void* desc, CacheView& v) {
  switch (layout) {
    case OL_LAYOUT_CONTIGUOUS:
      return view_contiguous(static_cast<const ol_kv_cache*>(desc), v);
    case OL_LAYOUT_PAGED:
      return view_paged(static_cast<const ol_paged_kv*>(desc), v);
    case OL_LAYOUT_INT4:
      return view_int4(static_cast<const ol_int4_kv*>(desc), v);
    default:
      return OL_ERR_UNSUPPORTED;
  }
}

// The buffer must not overlap any cache storage range.
ol_status no_overlap(const CacheView& v, const void* p, size_t bytes) {
  if (!p || bytes == 0) return OL_OK;
  Range r = range_of(p, bytes);
  for (int i = 0; i < v.nranges; ++i)
    if (overlaps(r, v.ranges[i])) return OL_ERR_ALIAS;
  return OL_OK;
}

ol_status writable(const CacheView& v, const void* updated) {
  if (!updated) return OL_ERR_NULL;
  if (updated != v.alias_ptr) return OL_ERR_ALIAS;
  if (v.access != OL_READ_WRITE) return OL_ERR_READONLY;
  return OL_OK;
}

// Paged validation: every page a row reads or writes is inside the pool; a
// page that a row appends into is referenced by no other row.
ol_status check_pages(const ol_paged_kv* c, const int32_t* lens_or_pos, int new_len, bool append,
                      int window) {
  const int S = c->page_size;
  std::vector<int> first_row(append ? c->num_pages : 0, -1);
  std::vector<char> shared(append ? c->num_pages : 0, 0);
  for (int b = 0; b < c->batch; ++b) {
    int lo, hi;
    if (append) {  // history [0, p) is read, [p, p + new_len) written
      lo = 0;
      hi = lens_or_pos[b] + new_len;
    } else {
      RowSplit rs = row_split(lens_or_pos[b], window, 1);
      lo = rs.lo;
      hi = rs.hi;
    }
    if (hi <= lo) continue;
    for (int pg = lo / S; pg <= (hi - 1) / S; ++pg) {
      int page = c->block_table_host[(size_t)b * c->max_pages + pg];
      if (page < 0 || page >= c->num_pages) return OL_ERR_PAGE;
      if (append) {
        if (first_row[page] == -1)
          first_row[page] = b;
        else if (first_row[page] != b)
          shared[page] = 1;
      }
    }
  }
  if (append)
    for (int b = 0; b < c->batch; ++b) {
      int p0 = lens_or_pos[b];
      for (int t = p0; t < p0 + new_len; ++t)
        if (shared[c->block_table_host[(size_t)b * c->max_pages + t / S]]) return OL_ERR_PAGE;
    }
  return OL_OK;
}

AttnParams base_params(const CacheView& v, int layout, const void* desc) {
  AttnParams p = {};
  p.layout = layout;
  p.dtype = v.dtype;
  p.batch = v.batch;
  p.kv_heads = v.kv_heads;
  p.head_dim = v.head_dim;
  p.capacity = v.capacity;
  if (layout == OL_LAYOUT_CONTIGUOUS) {
    p.cache = static_cast<const ol_kv_cache*>(desc)->data;
  } else if (layout == OL_LAYOUT_PAGED) {
    const ol_paged_kv* c = static_cast<const ol_paged_kv*>(desc);
    p.pool = c->data;
    p.block_table = c->block_table;
    p.num_pages = c->num_pages;
    p.page_size = c->page_size;
    p.max_pages = c->max_pages;
  } else if (layout == OL_LAYOUT_HPAGED) {
    const ol_hpaged_kv* c = static_cast<const ol_hpaged_kv*>(desc);
    p.pool = c->pool;
    p.block_table = c->block_table;
    p.num_pages = c->num_pages;
    p.page_size = c->page_size;
    p.max_pages = c->max_pages;
    p.page_fmt = c->formats;
  } else {
    const ol_int4_kv* c = static_cast<const ol_int4_kv*>(desc);
    p.codes = c->codes;
    p.scales = c->scales;
    p.zps = c->zps;
    p.quant_mode = c->quant_mode;
    p.fixed_scale = c->fixed_scale;
    p.fixed_zp = c->fixed_zp;
  }
  return p;
}

// Shared path of every attention-bearing call.
// ----------------------------------------------------- storage statistics

thread_local ol_stats t_last = {};
thread_local ol_stats t_total = {};

void record(const ol_stats& s) {
  t_last = s;
  t_total.calls += s.calls;
  t_total.storage_allocations += s.storage_allocations;
  t_total.storage_allocated_bytes += s.storage_allocated_bytes;
  t_total.storage_prefix_copied_bytes += s.storage_prefix_copied_bytes;
  t_total.storage_append_copied_bytes += s.storage_append_copied_bytes;
  t_total.storage_reuse_count += s.storage_reuse_count;
  t_total.dequantized_bytes += s.dequantized_bytes;
  t_total.attended_tokens += s.attended_tokens;
  t_total.kv_payload_bytes_read += s.kv_payload_bytes_read;
  t_total.workspace_bytes = std::max(t_total.workspace_bytes, s.workspace_bytes);
}

// Stored payload bytes of one token of one kv head in one plane (K or V).
int64_t token_payload(const CacheView& v) {
  return v.layout == OL_LAYOUT_INT4 ? v.head_dim / 2 + (v.head_dim / 32) * 2 + v.head_dim / 64
                                    : (int64_t)v.head_dim * (int64_t)elt_bytes(v.dtype);
}

// An append of new_len tokens to every row: written in place, nothing else copied.
void record_append(const CacheView& v, int new_len) {
  ol_stats s = {};
  s.calls = 1;
  s.storage_append_copied_bytes = 2ll * v.batch * v.kv_heads * new_len * token_payload(v);
  s.storage_reuse_count = new_len > 0 && v.batch > 0 ? 2 : 0;
  record(s);
}

// An attention call (with the fused append when `append`): history read from
// the cache is the visible range minus the current token when that one comes
// from new_kv.
void record_attention(const CacheView& v, const int32_t* lens_host, int window, int append, int cur_from_new,
                      size_t ws_need, int nq) {
  ol_stats s = {};
  s.calls = 1;
  int64_t visible = 0, hist = 0;
  for (int z = 0; z < nq; ++z)  // query token z of a chunk sees up to lens - nq + z
    for (int b = 0; b < v.batch; ++b) {
      const RowSplit rs = row_split(lens_host[b] - (nq - 1 - z), window < 0 ? -1 : window, 16);
      const int vis = rs.hi - rs.lo;
      visible += vis;
      // tokens taken from new_kv instead of the cache: the chunk's first z + 1
      const int fresh = cur_from_new ? std::min(z + 1, vis) : 0;
      hist += vis - fresh;
    }
  s.attended_tokens = visible * v.kv_heads;
  s.kv_payload_bytes_read = 2 * hist * v.kv_heads * token_payload(v);
  if (v.layout == OL_LAYOUT_INT4) s.dequantized_bytes = 2 * hist * v.kv_heads * v.head_dim * 4;
  if (append) {
    s.storage_append_copied_bytes = 2ll * v.batch * v.kv_heads * token_payload(v);
    s.storage_reuse_count = v.batch > 0 ? 2 : 0;
  }
  s.workspace_bytes = (int64_t)ws_need;
  record(s);
}

// Heterogeneous pages: payload and dequantized bytes follow each page's formats.
// read_lo/read_hi: the tokens read from the cache per row; nf: formats of the
// pages a fused append starts (or NULL); append_pos: the fused append's
// position per row (or NULL).
void record_hpaged(const ol_hpaged_kv* c, const int32_t* read_lo, const int32_t* read_hi, int nranges,
                   int64_t attended, const int32_t* append_pos, int new_len, const ol_page_format* nf,
                   size_t ws_need) {
  ol_stats s = {};
  s.calls = 1;
  const int S = c->page_size, D = c->head_dim;
  auto plane_bytes = [&](const ol_plane_format& f, int64_t n) {
    s.kv_payload_bytes_read += n * (int64_t)fmt_row_bytes(f.format, D);
    if (fmt_affine(f.format)) s.dequantized_bytes += n * D * 4;
  };
  for (int r = 0; read_lo && r < c->batch * nranges; ++r) {
    const int b = r % c->batch;
    for (int t = read_lo[r]; t < read_hi[r];) {
      const int end = std::min(read_hi[r], (t / S + 1) * S);
      const ol_page_format& f = c->formats_host[c->block_table_host[(size_t)b * c->max_pages + t / S]];
      plane_bytes(f.k, (int64_t)(end - t) * c->kv_heads);
      plane_bytes(f.v, (int64_t)(end - t) * c->kv_heads);
      t = end;
    }
  }
  for (int b = 0; append_pos && b < c->batch; ++b)
    for (int t = append_pos[b]; t < append_pos[b] + new_len; ++t) {
      const ol_page_format& f = hpaged_token_format(c, b, t, append_pos[b], *nf);
      s.storage_append_copied_bytes +=
          (int64_t)c->kv_heads * (int64_t)(fmt_row_bytes(f.k.format, D) + fmt_row_bytes(f.v.format, D));
    }
  if (append_pos && new_len > 0 && c->batch > 0) s.storage_reuse_count = 2;
  s.attended_tokens = attended * c->kv_heads;
  s.workspace_bytes = (int64_t)ws_need;
  record(s);
}

// The INT4 tensor-core kernel takes the step: a chunked step's query tokens
// share a CTA as extra MMA columns, 8 / group of them (p.tq).
bool int4_fast_path(AttnParams& p) {
  p.tq = p.nq > 1 ? std::max(1, std::min(p.nq, 8 / std::max(1, p.group))) : 1;
  return fast_int4_supported(p);
}

// The heterogeneous-page tensor-core kernel takes the step (query tokens of a
// chunked step as extra columns, as for INT4).
bool hpaged_fast_path(AttnParams& p) {
  p.tq = p.nq > 1 ? std::max(1, std::min(p.nq, 8 / std::max(1, p.group))) : 1;
  return fast_hpaged_supported(p);
}

// nq > 1: a chunked step's attention (query tokens z = 0..nq-1 per row, token z
// at position lens - nq + z; q and y are [B, Hq, nq, D]). check_only: stop
// after validation (nothing recorded, nothing launched).
ol_status run_attention(int layout, const void* desc, const CacheView& v, const void* q, int q_heads,
                        const int32_t* lens_host, const int32_t* lens_dev, const void* new_kv, int append,
                        int cur_from_new, float scale, int window, void* out, int out_dtype, void* workspace,
                        size_t ws_bytes, cudaStream_t stream, int nq = 1, bool check_only = false,
                        const ol_page_format* new_fmt = nullptr, bool inputs_ready = false) {
  if (!q || !lens_host || !lens_dev || !out || !workspace) return OL_ERR_NULL;
  if (q_heads <= 0 || q_heads % v.kv_heads != 0) return OL_ERR_SHAPE;
  if (v.head_dim > 256) return OL_ERR_UNSUPPORTED;
  if (!valid_dtype(out_dtype)) return OL_ERR_DTYPE;
  if (!aligned16(q) || !aligned16(lens_dev) || !aligned16(out) || !aligned16(workspace) ||
      (new_kv && !aligned16(new_kv)))
    return OL_ERR_ALIGN;
  const int D = v.head_dim;
  const int min_len = nq > 1 ? nq : (append ? 1 : 0);
  for (int b = 0; b < v.batch; ++b) {
    if (lens_host[b] < min_len || lens_host[b] > v.capacity) return OL_ERR_CAPACITY;
  }
  const size_t in_elt = v.layout == OL_LAYOUT_INT4 ? 2 : elt_bytes(v.dtype);
  const size_t q_bytes = (size_t)v.batch * q_heads * nq * D * in_elt;
  const size_t out_bytes = (size_t)v.batch * q_heads * nq * D * elt_bytes(out_dtype);
  const size_t kv_bytes = 2ull * v.batch * v.kv_heads * nq * D * in_elt;
  const size_t need = workspace_bytes(v.batch, q_heads, v.kv_heads, D, nq);
  if (ws_bytes < need) return OL_ERR_WORKSPACE;
  ol_status st;
  if ((st = no_overlap(v, q, q_bytes)) != OL_OK) return st;
  if ((st = no_overlap(v, out, out_bytes)) != OL_OK) return st;
  if ((st = no_overlap(v, new_kv, kv_bytes)) != OL_OK) return st;
  if ((st = no_overlap(v, workspace, need)) != OL_OK) return st;
  if ((st = no_overlap(v, lens_dev, sizeof(int32_t) * v.batch)) != OL_OK) return st;
  if (overlaps(range_of(out, out_bytes), range_of(q, q_bytes)) ||
      overlaps(range_of(out, out_bytes), range_of(workspace, need)) ||
      (new_kv && overlaps(range_of(out, out_bytes), range_of(new_kv, kv_bytes))))
    return OL_ERR_ALIAS;
  if (layout == OL_LAYOUT_PAGED) {
    const ol_paged_kv* c = static_cast<const ol_paged_kv*>(desc);
    if ((st = no_overlap(v, c->block_table, sizeof(int32_t) * (size_t)c->batch * c->max_pages)) != OL_OK) return st;
    if (append) {
      std::vector<int32_t> pos(v.batch);
      for (int b = 0; b < v.batch; ++b) pos[b] = lens_host[b] - 1;
      if ((st = check_pages(c, pos.data(), 1, true, window)) != OL_OK) return st;
    } else if ((st = check_pages(c, lens_host, 0, false, window < 0 ? -1 : window + nq - 1)) != OL_OK) {
      return st;
    }
  }
  std::vector<int32_t> read_lo, read_hi, append_pos;
  if (layout == OL_LAYOUT_HPAGED) {
    const ol_hpaged_kv* c = static_cast<const ol_hpaged_kv*>(desc);
    if (nq != 1 && append) return OL_ERR_UNSUPPORTED;  // the fused append is the decode step's
    if ((st = no_overlap(v, c->block_table, sizeof(int32_t) * (size_t)c->batch * c->max_pages)) != OL_OK) return st;
    const int wq = window < 0 ? -1 : window;              // one query token's window
    const int wu = window < 0 ? -1 : window + nq - 1;     // the union of a chunk's query tokens' ranges
    const ol_paged_kv k = paged_shape_of(c);
    if (append) {
      if (!new_fmt) return OL_ERR_NULL;
      if (!valid_page_format(*new_fmt)) return OL_ERR_SHAPE;
      append_pos.resize(v.batch);
      for (int b = 0; b < v.batch; ++b) append_pos[b] = lens_host[b] - 1;
      if ((st = check_pages(&k, append_pos.data(), 1, true, window)) != OL_OK) return st;
    } else if ((st = check_pages(&k, lens_host, 0, false, wu)) != OL_OK) {
      return st;
    }
    // tokens taken from new_kv instead of the pages: the decode step's current
    // token, or a chunk's tokens (query token z sees the first z + 1 of them)
    std::vector<int32_t> union_hi(v.batch);
    for (int b = 0; b < v.batch; ++b) {
      const RowSplit rs = row_split(lens_host[b], wu, 1);
      union_hi[b] = rs.hi - (cur_from_new ? std::min(nq, rs.hi - rs.lo) : 0);
    }
    if ((st = check_hpaged_formats(c, lens_host, wu, union_hi.data(), append ? append_pos.data() : nullptr,
                                   append ? 1 : 0)) != OL_OK)
      return st;
    read_lo.resize((size_t)v.batch * nq);
    read_hi.resize((size_t)v.batch * nq);
    int64_t attended = 0;
    for (int z = 0; z < nq; ++z)
      for (int b = 0; b < v.batch; ++b) {
        const RowSplit rs = row_split(lens_host[b] - (nq - 1 - z), wq, 1);
        read_lo[(size_t)z * v.batch + b] = rs.lo;
        read_hi[(size_t)z * v.batch + b] = rs.hi - (cur_from_new ? std::min(z + 1, rs.hi - rs.lo) : 0);
        attended += rs.hi - rs.lo;
      }
    if ((st = check_owner(v.ranges, v.nranges, v.owner)) != OL_OK) return st;
    if (check_only) return OL_OK;
    record_hpaged(c, read_lo.data(), read_hi.data(), nq, attended, append ? append_pos.data() : nullptr, 1, new_fmt,
                  need);
  } else {
    if ((st = check_owner(v.ranges, v.nranges, v.owner)) != OL_OK) return st;
    if (check_only) return OL_OK;
    record_attention(v, lens_host, window, append, cur_from_new, need, nq);
  }
  if (fault_injected()) return OL_ERR_INJECTED;

  AttnParams p = base_params(v, layout, desc);
  p.q_heads = q_heads;
  p.group = q_heads / v.kv_heads;
  p.q = q;
  p.lens = lens_dev;
  p.new_kv = new_kv;
  p.append = append;
  p.cur_from_new = cur_from_new;
  p.scale = scale > 0.f ? scale : 1.0f / std::sqrt((float)D);
  p.scale_log2 = p.scale * 1.4426950408889634f;
  p.window_q = window < 0 ? -1 : window;
  p.window = window < 0 ? -1 : window + nq - 1;  // the union of the query tokens' ranges
  p.nq = nq;
  if (new_fmt) p.new_fmt = *new_fmt;
  p.out = out;
  p.out_dtype = out_dtype;
  p.inline_lens = v.batch <= kInlineRows ? 1 : 0;
  if (p.inline_lens)
    for (int b = 0; b < v.batch; ++b) p.lens_inline[b] = lens_host[b];
  p.early = (v.history_stable && p.inline_lens) ? 1 : 0;
  p.inputs_ready = inputs_ready ? 1 : 0;
  char* ws = static_cast<char*>(workspace);
  p.status = reinterpret_cast<int32_t*>(ws);
  p.counters = reinterpret_cast<uint32_t*>(ws + kStatusBytes);
  p.partials = reinterpret_cast<float*>(ws + partials_offset(v.batch, v.kv_heads, nq));

  const int sms = sm_count_cached();
  cudaError_t e;
  p.tq = 1;
  if (layout != OL_LAYOUT_INT4 && fast_bf16_supported(p)) {
    // a chunk's query tokens share a CTA as extra MMA columns: 8 / group of them
    if (nq > 1) p.tq = std::max(1, std::min(nq, 8 / p.group));
    plan_fast(p, lens_host, sms);
    order_rows(p, lens_host);
    e = launch_fast_bf16(p, stream);
  } else if (layout == OL_LAYOUT_INT4 && int4_fast_path(p)) {
    plan_fast(p, lens_host, sms);
    order_rows(p, lens_host);
    e = launch_fast_int4(p, stream);
  } else if (layout == OL_LAYOUT_HPAGED && hpaged_fast_path(p) && !tune().generic) {
    plan_splits(p, lens_host, (long long)sms * fast_hpaged_ctas_per_sm(p.nq > 1) * tune().hp_waves, 1);
    order_rows(p, lens_host);
    p.variant = 0;
    e = launch_fast_hpaged(p, stream);
  } else {
    p.tq = 1;  // the CUDA-core kernel serves one query token per grid slice
    plan_splits(p, lens_host, (long long)sms * 4, 1);
    order_rows(p, lens_host);
    p.variant = 0;
    e = launch_generic_attention(p, stream);
  }
  return e == cudaSuccess ? OL_OK : OL_ERR_CUDA;
}

}  // namespace

ol_status decode_step_impl(int32_t layout, const void* cache_desc, void* updated, const void* q, int32_t q_heads,
                           const void* new_kv, const int32_t* lens_host, const int32_t* lens_dev, float scale,
                           int32_t window, void* out, int32_t out_dtype, void* workspace, size_t ws_bytes,
                           ol_stream stream, bool check_only) {
  CacheView v;
  ol_status st = view_of(layout, cache_desc, v);
  if (st != OL_OK) return st;
  if ((st = writable(v, updated)) != OL_OK) return st;
  if (!new_kv) return OL_ERR_NULL;
  return run_attention(layout, cache_desc, v, q, q_heads, lens_host, lens_dev, new_kv, 1, 1, scale, window, out,
                       out_dtype, workspace, ws_bytes, static_cast<cudaStream_t>(stream), 1, check_only);
}

}  // namespace ol

using namespace ol;

extern "C" {

const char* ol_status_string(ol_status s) {
  switch (s) {
    case OL_OK: return "OL_OK";
    case OL_ERR_NULL: return "OL_ERR_NULL: a required pointer is NULL";
    case OL_ERR_ALIAS: return "OL_ERR_ALIAS: updated pointer differs from the cache, or a buffer overlaps the cache";
    case OL_ERR_READONLY: return "OL_ERR_READONLY: the cache descriptor is read-only";
    case OL_ERR_CAPACITY: return "OL_ERR_CAPACITY: position + length exceeds the cache capacity";
    case OL_ERR_SHAPE: return "OL_ERR_SHAPE: inconsistent or invalid sizes";
    case OL_ERR_DTYPE: return "OL_ERR_DTYPE: unsupported dtype";
    case OL_ERR_BUSY: return "OL_ERR_BUSY: the cache is bound by another owner";
    case OL_ERR_WORKSPACE: return "OL_ERR_WORKSPACE: workspace missing or too small";
    case OL_ERR_CUDA: return "OL_ERR_CUDA: a CUDA call failed";
    case OL_ERR_UNSUPPORTED: return "OL_ERR_UNSUPPORTED: not implemented for these sizes";
    case OL_ERR_INJECTED: return "OL_ERR_INJECTED: host fault injection after validation";
    case OL_ERR_PAGE: return "OL_ERR_PAGE: invalid block-table entry or shared append page";
    case OL_ERR_ALIGN: return "OL_ERR_ALIGN: device pointer not 16-byte aligned";
  }
  return "unknown ol_status";
}

int32_t ol_version(void) { return 100; }

ol_status ol_last_call_stats(ol_stats* out) {
  if (!out) return OL_ERR_NULL;
  *out = t_last;
  return OL_OK;
}

ol_status ol_total_stats(ol_stats* out) {
  if (!out) return OL_ERR_NULL;
  *out = t_total;
  return OL_OK;
}

void ol_reset_stats(void) {
  t_last = ol_stats{};
  t_total = ol_stats{};
}

size_t ol_workspace_size(int32_t batch, int32_t q_heads, int32_t kv_heads, int32_t head_dim) {
  if (batch < 0 || kv_heads <= 0 || q_heads <= 0 || q_heads % kv_heads != 0 || head_dim <= 0) return 0;
  return workspace_bytes(batch, q_heads, kv_heads, head_dim);
}

ol_status ol_workspace_init(void* workspace, size_t ws_bytes, ol_stream stream) {
  if (!workspace) return OL_ERR_NULL;
  return cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess ? OL_OK
                                                                                                    : OL_ERR_CUDA;
}

ol_status ol_workspace_status(void* workspace, int32_t* status_out, ol_stream stream) {
  if (!workspace || !status_out) return OL_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return OL_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return OL_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof v, s) != cudaSuccess) return OL_ERR_CUDA;
  *status_out = v;
  return OL_OK;
}

ol_status ol_cache_bind(const void* base, size_t bytes, uint64_t owner) {
  if (!base || bytes == 0) return OL_ERR_NULL;
  Range r = range_of(base, bytes);
  std::lock_guard<std::mutex> lk(g_bind_mu);
  for (const Binding& bd : g_bindings)
    if (overlaps(r, Range{bd.lo, bd.hi}) && bd.owner != owner) return OL_ERR_BUSY;
  for (Binding& bd : g_bindings)
    if (bd.lo == r.lo && bd.owner == owner) {
      bd.hi = r.hi > bd.hi ? r.hi : bd.hi;
      return OL_OK;
    }
  g_bindings.push_back({r.lo, r.hi, owner});
  return OL_OK;
}

ol_status ol_cache_unbind(const void* base, uint64_t owner) {
  if (!base) return OL_ERR_NULL;
  uintptr_t a = reinterpret_cast<uintptr_t>(base);
  std::lock_guard<std::mutex> lk(g_bind_mu);
  for (size_t i = 0; i < g_bindings.size(); ++i)
    if (g_bindings[i].lo == a) {
      if (g_bindings[i].owner != owner) return OL_ERR_BUSY;
      g_bindings.erase(g_bindings.begin() + (long)i);
      return OL_OK;
    }
  return OL_OK;
}

static ol_status append_common(const CacheView& v, const void* updated, const void* values, int32_t new_len,
                               const int32_t* positions_host, const int32_t* positions_dev) {
  ol_status st;
  if ((st = writable(v, updated)) != OL_OK) return st;
  if (!values || !positions_host || !positions_dev) return OL_ERR_NULL;
  if (new_len < 0) return OL_ERR_SHAPE;
  if (!aligned16(values) || !aligned16(positions_dev)) return OL_ERR_ALIGN;
  for (int b = 0; b < v.batch; ++b)
    if (positions_host[b] < 0 || (long long)positions_host[b] + new_len > v.capacity) return OL_ERR_CAPACITY;
  const size_t in_elt = v.layout == OL_LAYOUT_INT4 ? 2 : elt_bytes(v.dtype);
  if ((st = no_overlap(v, values, 2ull * v.batch * v.kv_heads * new_len * v.head_dim * in_elt)) != OL_OK) return st;
  if ((st = no_overlap(v, positions_dev, sizeof(int32_t) * v.batch)) != OL_OK) return st;
  return OL_OK;
}

static ol_status launch_append_view(const CacheView& v, int layout, const void* desc, const void* values,
                                    int32_t new_len, const int32_t* positions_dev, cudaStream_t s,
                                    int positions_are_lens = 0) {
  AppendParams p = {};
  p.positions_are_lens = positions_are_lens;
  p.layout = layout;
  p.dtype = v.dtype;
  p.batch = v.batch;
  p.kv_heads = v.kv_heads;
  p.head_dim = v.head_dim;
  p.capacity = v.capacity;
  p.new_len = new_len;
  p.values = values;
  p.positions = positions_dev;
  if (layout == OL_LAYOUT_CONTIGUOUS) {
    p.cache = static_cast<const ol_kv_cache*>(desc)->data;
  } else if (layout == OL_LAYOUT_PAGED) {
    const ol_paged_kv* c = static_cast<const ol_paged_kv*>(desc);
    p.pool = c->data;
    p.block_table = c->block_table;
    p.num_pages = c->num_pages;
    p.page_size = c->page_size;
    p.max_pages = c->max_pages;
  } else {
    const ol_int4_kv* c = static_cast<const ol_int4_kv*>(desc);
    p.codes = c->codes;
    p.scales = c->scales;
    p.zps = c->zps;
    p.quant_mode = c->quant_mode;
    p.fixed_scale = c->fixed_scale;
    p.fixed_zp = c->fixed_zp;
  }
  return launch_append(p, s) == cudaSuccess ? OL_OK : OL_ERR_CUDA;
}

ol_status ol_cache_update_rows(const ol_kv_cache* cache, void* updated_cache, const void* values, int32_t new_len,
                               const int32_t* positions_host, const int32_t* positions_dev, ol_stream stream) {
  CacheView v;
  ol_status st = view_contiguous(cache, v);
  if (st != OL_OK) return st;
  if ((st = append_common(v, updated_cache, values, new_len, positions_host, positions_dev)) != OL_OK) return st;
  if ((st = check_owner(v.ranges, v.nranges, v.owner)) != OL_OK) return st;
  record_append(v, new_len);
  if (fault_injected()) return OL_ERR_INJECTED;
  return launch_append_view(v, OL_LAYOUT_CONTIGUOUS, cache, values, new_len, positions_dev,
                            static_cast<cudaStream_t>(stream));
}

ol_status ol_cache_update(const ol_kv_cache* cache, void* updated_cache, const void* values, int32_t new_len,
                          int64_t position, ol_stream stream) {
  // One position for every row (the INT64 scalar of CacheUpdate), passed by value.
  CacheView v;
  ol_status st = view_contiguous(cache, v);
  if (st != OL_OK) return st;
  if (position < 0 || position > (int64_t)v.capacity) return OL_ERR_CAPACITY;
  if ((st = writable(v, updated_cache)) != OL_OK) return st;
  if (!values) return OL_ERR_NULL;
  if (new_len < 0) return OL_ERR_SHAPE;
  if (!aligned16(values)) return OL_ERR_ALIGN;
  if (position + new_len > (int64_t)v.capacity) return OL_ERR_CAPACITY;
  if ((st = no_overlap(v, values, 2ull * v.batch * v.kv_heads * new_len * v.head_dim * elt_bytes(v.dtype))) != OL_OK)
    return st;
  if ((st = check_owner(v.ranges, v.nranges, v.owner)) != OL_OK) return st;
  record_append(v, new_len);
  if (fault_injected()) return OL_ERR_INJECTED;
  AppendParams p = {};
  p.layout = OL_LAYOUT_CONTIGUOUS;
  p.dtype = v.dtype;
  p.batch = v.batch;
  p.kv_heads = v.kv_heads;
  p.head_dim = v.head_dim;
  p.capacity = v.capacity;
  p.new_len = new_len;
  p.values = values;
  p.positions = nullptr;
  p.cache = cache->data;
  p.scalar_position = static_cast<int32_t>(position);
  return launch_append(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? OL_OK : OL_ERR_CUDA;
}

ol_status ol_paged_cache_update(const ol_paged_kv* kv, void* updated_pool, const void* values, int32_t new_len,
                                const int32_t* positions_host, const int32_t* positions_dev, ol_stream stream) {
  CacheView v;
  ol_status st = view_paged(kv, v);
  if (st != OL_OK) return st;
  if ((st = append_common(v, updated_pool, values, new_len, positions_host, positions_dev)) != OL_OK) return st;
  if ((st = no_overlap(v, kv->block_table, sizeof(int32_t) * (size_t)kv->batch * kv->max_pages)) != OL_OK) return st;
  if ((st = check_pages(kv, positions_host, new_len, true, -1)) != OL_OK) return st;
  if ((st = check_owner(v.ranges, v.nranges, v.owner)) != OL_OK) return st;
  record_append(v, new_len);
  if (fault_injected()) return OL_ERR_INJECTED;
  return launch_append_view(v, OL_LAYOUT_PAGED, kv, values, new_len, positions_dev, static_cast<cudaStream_t>(stream));
}

ol_status ol_int4kv_append(const ol_int4_kv* cache, void* updated_codes, const void* values_bf16,
                           const int32_t* positions_host, const int32_t* positions_dev, ol_stream stream) {
  CacheView v;
  ol_status st = view_int4(cache, v);
  if (st != OL_OK) return st;
  if ((st = append_common(v, updated_codes, values_bf16, 1, positions_host, positions_dev)) != OL_OK) return st;
  if ((st = check_owner(v.ranges, v.nranges, v.owner)) != OL_OK) return st;
  record_append(v, 1);
  if (fault_injected()) return OL_ERR_INJECTED;
  return launch_append_view(v, OL_LAYOUT_INT4, cache, values_bf16, 1, positions_dev, static_cast<cudaStream_t>(stream));
}

ol_status ol_decode_attention(const ol_kv_cache* cache, const void* q, int32_t q_heads, const int32_t* lens_host,
                              const int32_t* lens_dev, float scale, int32_t window, void* out, int32_t out_dtype,
                              void* workspace, size_t ws_bytes, ol_stream stream) {
  CacheView v;
  ol_status st = view_contiguous(cache, v);
  if (st != OL_OK) return st;
  return run_attention(OL_LAYOUT_CONTIGUOUS, cache, v, q, q_heads, lens_host, lens_dev, nullptr, 0, 0, scale, window,
                       out, out_dtype, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

ol_status ol_paged_decode_attention(const ol_paged_kv* kv, const void* q, int32_t q_heads, const int32_t* lens_host,
                                    const int32_t* lens_dev, float scale, int32_t window, void* out,
                                    int32_t out_dtype, void* workspace, size_t ws_bytes, ol_stream stream) {
  CacheView v;
  ol_status st = view_paged(kv, v);
  if (st != OL_OK) return st;
  return run_attention(OL_LAYOUT_PAGED, kv, v, q, q_heads, lens_host, lens_dev, nullptr, 0, 0, scale, window, out,
                       out_dtype, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

ol_status ol_int4kv_decode_attention(const ol_int4_kv* cache, const void* q, int32_t q_heads,
                                     const int32_t* lens_host, const int32_t* lens_dev, const void* cur_kv,
                                     float scale, int32_t window, void* out, int32_t out_dtype, void* workspace,
                                     size_t ws_bytes, ol_stream stream) {
  CacheView v;
  ol_status st = view_int4(cache, v);
  if (st != OL_OK) return st;
  if (cur_kv && lens_host)
    for (int b = 0; b < v.batch; ++b)
      if (lens_host[b] < 1) return OL_ERR_CAPACITY;
  return run_attention(OL_LAYOUT_INT4, cache, v, q, q_heads, lens_host, lens_dev, cur_kv, 0, cur_kv ? 1 : 0, scale,
                       window, out, out_dtype, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

ol_status ol_decode_step(int32_t layout, const void* cache_desc, void* updated, const void* q, int32_t q_heads,
                         const void* new_kv, const int32_t* lens_host, const int32_t* lens_dev, float scale,
                         int32_t window, void* out, int32_t out_dtype, void* workspace, size_t ws_bytes,
                         ol_stream stream) {
  return ol::decode_step_impl(layout, cache_desc, updated, q, q_heads, new_kv, lens_host, lens_dev, scale, window,
                              out, out_dtype, workspace, ws_bytes, stream, false);
}

// Staging offsets inside the workspace for ol_decode_step_host, after the
// bytes ol_decode_step needs; every buffer 256-byte aligned and sized for
// 4-byte elements.
struct HostStaging {
  size_t q, kv, lens, out, total;
};
static HostStaging host_staging(int32_t batch, int32_t q_heads, int32_t kv_heads, int32_t head_dim) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  HostStaging h;
  h.q = up(workspace_bytes(batch, q_heads, kv_heads, head_dim));
  h.kv = h.q + up((size_t)batch * q_heads * head_dim * 4);
  h.lens = h.kv + up(2ull * batch * kv_heads * head_dim * 4);
  h.out = h.lens + up((size_t)batch * 4);
  h.total = h.out + up((size_t)batch * q_heads * head_dim * 4);
  return h;
}

size_t ol_workspace_size_chunk(int32_t batch, int32_t q_heads, int32_t kv_heads, int32_t head_dim,
                               int32_t new_len) {
  if (batch < 0 || kv_heads <= 0 || q_heads <= 0 || q_heads % kv_heads != 0 || head_dim <= 0 || new_len < 1)
    return 0;
  return workspace_bytes(batch, q_heads, kv_heads, head_dim, new_len);
}

ol_status ol_chunk_step(int32_t layout, const void* cache_desc, void* updated, const void* q, int32_t q_heads,
                        int32_t new_len, const void* new_kv, const int32_t* lens_host, const int32_t* lens_dev,
                        float scale, int32_t window, void* out, int32_t out_dtype, void* workspace, size_t ws_bytes,
                        ol_stream stream) {
  CacheView v;
  ol_status st = view_of(layout, cache_desc, v);
  if (st != OL_OK) return st;
  // INT4: the chunk's tokens are attended uncompressed from new_kv, then encoded
  const bool int4 = layout == OL_LAYOUT_INT4;
  if (new_len < 1) return OL_ERR_SHAPE;
  if (!lens_host) return OL_ERR_NULL;
  // the append writes positions lens - new_len .. lens - 1 of every row
  std::vector<int32_t> pos(v.batch);
  for (int b = 0; b < v.batch; ++b) {
    if (lens_host[b] < new_len || lens_host[b] > v.capacity) return OL_ERR_CAPACITY;
    pos[b] = lens_host[b] - new_len;
  }
  if ((st = append_common(v, updated, new_kv, new_len, pos.data(), lens_dev)) != OL_OK) return st;
  if (layout == OL_LAYOUT_PAGED) {
    const ol_paged_kv* c = static_cast<const ol_paged_kv*>(cache_desc);
    if ((st = no_overlap(v, c->block_table, sizeof(int32_t) * (size_t)c->batch * c->max_pages)) != OL_OK) return st;
    if ((st = check_pages(c, pos.data(), new_len, true, -1)) != OL_OK) return st;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // every check of the attention first: an error return means nothing was written
  if ((st = run_attention(layout, cache_desc, v, q, q_heads, lens_host, lens_dev, int4 ? new_kv : nullptr, 0,
                          int4 ? 1 : 0, scale, window, out, out_dtype, workspace, ws_bytes, s, new_len, true)) != OL_OK)
    return st;
  const size_t in_elt = elt_bytes(v.dtype);
  if ((st = no_overlap(v, new_kv, 2ull * v.batch * v.kv_heads * new_len * v.head_dim * in_elt)) != OL_OK) return st;
  if (overlaps(range_of(out, (size_t)v.batch * q_heads * new_len * v.head_dim * elt_bytes(out_dtype)),
               range_of(new_kv, 2ull * v.batch * v.kv_heads * new_len * v.head_dim * in_elt)))
    return OL_ERR_ALIAS;
  if ((st = check_owner(v.ranges, v.nranges, v.owner)) != OL_OK) return st;
  if (fault_injected()) return OL_ERR_INJECTED;
  if (int4) {
    st = run_attention(layout, cache_desc, v, q, q_heads, lens_host, lens_dev, new_kv, 0, 1, scale, window, out,
                       out_dtype, workspace, ws_bytes, s, new_len);
    if (st == OL_OK) st = launch_append_view(v, layout, cache_desc, new_kv, new_len, lens_dev, s, 1);
  } else {
    if ((st = launch_append_view(v, layout, cache_desc, new_kv, new_len, lens_dev, s, 1)) != OL_OK) return st;
    st = run_attention(layout, cache_desc, v, q, q_heads, lens_host, lens_dev, nullptr, 0, 0, scale, window, out,
                       out_dtype, workspace, ws_bytes, s, new_len);
  }
  // the call's one record: the attention's counts (recorded by run_attention) and the append's
  const int64_t appended = 2ll * v.batch * v.kv_heads * new_len * token_payload(v);
  for (ol_stats* r : {&t_last, &t_total}) {
    r->storage_append_copied_bytes += appended;
    r->storage_reuse_count += v.batch > 0 ? 2 : 0;
  }
  return st;
}

size_t ol_workspace_size_host(int32_t batch, int32_t q_heads, int32_t kv_heads, int32_t head_dim) {
  if (batch < 0 || kv_heads <= 0 || q_heads <= 0 || q_heads % kv_heads != 0 || head_dim <= 0) return 0;
  return host_staging(batch, q_heads, kv_heads, head_dim).total;
}

// The device address of page-locked host memory mapped into the device's
// address space (cudaHostAlloc'd, or registered with mapping), 16-byte
// aligned; nullptr for any other pointer (pageable memory, device memory).
static void* mapped_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the error the query left behind
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer || !aligned16(a.devicePointer)) return nullptr;
  return a.devicePointer;
}

ol_status ol_decode_step_host(int32_t layout, const void* cache_desc, void* updated, const void* q_host,
                              int32_t q_heads, const void* new_kv_host, const int32_t* lens_host, float scale,
                              int32_t window, void* out_host, int32_t out_dtype, void* workspace, size_t ws_bytes,
                              ol_stream stream) {
  CacheView v;
  ol_status st = view_of(layout, cache_desc, v);
  if (st != OL_OK) return st;
  if ((st = writable(v, updated)) != OL_OK) return st;
  if (!q_host || !new_kv_host || !lens_host || !out_host || !workspace) return OL_ERR_NULL;
  if (q_heads <= 0 || q_heads % v.kv_heads != 0) return OL_ERR_SHAPE;
  if (!valid_dtype(out_dtype)) return OL_ERR_DTYPE;
  if (!aligned16(workspace)) return OL_ERR_ALIGN;
  const HostStaging h = host_staging(v.batch, q_heads, v.kv_heads, v.head_dim);
  if (ws_bytes < h.total) return OL_ERR_WORKSPACE;
  if ((st = no_overlap(v, workspace, h.total)) != OL_OK) return st;
  for (int b = 0; b < v.batch; ++b)
    if (lens_host[b] < 1 || lens_host[b] > v.capacity) return OL_ERR_CAPACITY;
  const size_t in_elt = v.layout == OL_LAYOUT_INT4 ? 2 : elt_bytes(v.dtype);
  const size_t q_bytes = (size_t)v.batch * q_heads * v.head_dim * in_elt;
  const size_t kv_bytes = 2ull * v.batch * v.kv_heads * v.head_dim * in_elt;
  const size_t out_bytes = (size_t)v.batch * q_heads * v.head_dim * elt_bytes(out_dtype);
  // y must not overlap the step's inputs, whichever way each buffer travels
  if (overlaps(range_of(out_host, out_bytes), range_of(q_host, q_bytes)) ||
      overlaps(range_of(out_host, out_bytes), range_of(new_kv_host, kv_bytes)))
    return OL_ERR_ALIAS;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Mapped page-locked buffers are used in place: the step's kernels load q
  // and the new K/V from host memory and store y there, over the CPU-GPU
  // link, with no copy-engine copy (a few microseconds of GPU time each, the
  // larger part of a small step). Other buffers go through the workspace's
  // staging area with stream-ordered copies.
  const void* q_in = mapped_host(q_host);
  const void* kv_in = mapped_host(new_kv_host);
  void* out_to = mapped_host(out_host);
  if (!q_in) {
    if (cudaMemcpyAsync(ws + h.q, q_host, q_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return OL_ERR_CUDA;
    q_in = ws + h.q;
  }
  if (!kv_in) {
    if (cudaMemcpyAsync(ws + h.kv, new_kv_host, kv_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return OL_ERR_CUDA;
    kv_in = ws + h.kv;
  }
  // the kernels take the lengths by value for batches of up to kInlineRows
  // rows and never read the device copy then
  if (v.batch > kInlineRows &&
      cudaMemcpyAsync(ws + h.lens, lens_host, sizeof(int32_t) * v.batch, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return OL_ERR_CUDA;
  // q and the new K/V are the caller's host data, written before this call, or
  // copies ordered before the launch: the kernels may read them before they
  // wait for the previous launch to complete
  st = run_attention(layout, cache_desc, v, q_in, q_heads, lens_host, reinterpret_cast<int32_t*>(ws + h.lens),
                     kv_in, 1, 1, scale, window, out_to ? out_to : ws + h.out, out_dtype, workspace, h.q, s, 1,
                     false, nullptr, /*inputs_ready=*/true);
  if (st != OL_OK || out_to) return st;
  return cudaMemcpyAsync(out_host, ws + h.out, out_bytes, cudaMemcpyDeviceToHost, s) == cudaSuccess ? OL_OK
                                                                                                 : OL_ERR_CUDA;
}

// ------------------------------------------------ heterogeneous paged cache

ol_status ol_hpaged_append(const ol_hpaged_kv* cache, void* updated, const void* values_bf16, int32_t new_len,
                           const int32_t* positions_host, const int32_t* positions_dev,
                           const ol_page_format* new_pages, ol_stream stream) {
  CacheView v;
  ol_status st = view_hpaged(cache, v);
  if (st != OL_OK) return st;
  if ((st = append_common(v, updated, values_bf16, new_len, positions_host, positions_dev)) != OL_OK) return st;
  if (!new_pages) return OL_ERR_NULL;
  if (!valid_page_format(*new_pages)) return OL_ERR_SHAPE;
  if ((st = no_overlap(v, cache->block_table, sizeof(int32_t) * (size_t)cache->batch * cache->max_pages)) != OL_OK)
    return st;
  const ol_paged_kv k = paged_shape_of(cache);
  if ((st = check_pages(&k, positions_host, new_len, true, -1)) != OL_OK) return st;
  if (new_len > 0 &&
      (st = check_hpaged_formats(cache, nullptr, -1, nullptr, positions_host, new_len)) != OL_OK)
    return st;
  if ((st = check_owner(v.ranges, v.nranges, v.owner)) != OL_OK) return st;
  record_hpaged(cache, nullptr, nullptr, 1, 0, positions_host, new_len, new_pages, 0);
  if (fault_injected()) return OL_ERR_INJECTED;
  AppendParams p = {};
  p.layout = OL_LAYOUT_HPAGED;
  p.dtype = OL_BF16;
  p.batch = v.batch;
  p.kv_heads = v.kv_heads;
  p.head_dim = v.head_dim;
  p.capacity = v.capacity;
  p.new_len = new_len;
  p.values = values_bf16;
  p.positions = positions_dev;
  p.pool = cache->pool;
  p.block_table = cache->block_table;
  p.num_pages = cache->num_pages;
  p.page_size = cache->page_size;
  p.max_pages = cache->max_pages;
  p.page_fmt = cache->formats;
  p.new_fmt = *new_pages;
  if (launch_hpaged_append(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return OL_ERR_CUDA;
  if (new_len > 0) hpaged_start_pages(cache, positions_host, new_len, *new_pages);
  return OL_OK;
}

ol_status ol_hpaged_decode_attention(const ol_hpaged_kv* cache, const void* q, int32_t q_heads,
                                     const int32_t* lens_host, const int32_t* lens_dev, const void* cur_kv,
                                     float scale, int32_t window, void* out, int32_t out_dtype, void* workspace,
                                     size_t ws_bytes, ol_stream stream) {
  CacheView v;
  ol_status st = view_hpaged(cache, v);
  if (st != OL_OK) return st;
  if (cur_kv && lens_host)
    for (int b = 0; b < v.batch; ++b)
      if (lens_host[b] < 1) return OL_ERR_CAPACITY;
  return run_attention(OL_LAYOUT_HPAGED, cache, v, q, q_heads, lens_host, lens_dev, cur_kv, 0, cur_kv ? 1 : 0,
                       scale, window, out, out_dtype, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

ol_status ol_hpaged_decode_step(const ol_hpaged_kv* cache, void* updated, const void* q, int32_t q_heads,
                                const void* new_kv, const ol_page_format* new_pages, const int32_t* lens_host,
                                const int32_t* lens_dev, float scale, int32_t window, void* out, int32_t out_dtype,
                                void* workspace, size_t ws_bytes, ol_stream stream) {
  CacheView v;
  ol_status st = view_hpaged(cache, v);
  if (st != OL_OK) return st;
  if ((st = writable(v, updated)) != OL_OK) return st;
  if (!new_kv || !new_pages) return OL_ERR_NULL;
  st = run_attention(OL_LAYOUT_HPAGED, cache, v, q, q_heads, lens_host, lens_dev, new_kv, 1, 1, scale, window, out,
                     out_dtype, workspace, ws_bytes, static_cast<cudaStream_t>(stream), 1, false, new_pages);
  if (st != OL_OK) return st;
  std::vector<int32_t> pos(v.batch);
  for (int b = 0; b < v.batch; ++b) pos[b] = lens_host[b] - 1;
  hpaged_start_pages(cache, pos.data(), 1, *new_pages);
  return OL_OK;
}

ol_status ol_hpaged_chunk_step(const ol_hpaged_kv* cache, void* updated, const void* q, int32_t q_heads,
                               int32_t new_len, const void* new_kv, const ol_page_format* new_pages,
                               const int32_t* lens_host, const int32_t* lens_dev, float scale, int32_t window,
                               void* out, int32_t out_dtype, void* workspace, size_t ws_bytes, ol_stream stream) {
  CacheView v;
  ol_status st = view_hpaged(cache, v);
  if (st != OL_OK) return st;
  if (new_len < 1) return OL_ERR_SHAPE;
  if (!lens_host || !new_pages) return OL_ERR_NULL;
  // the append writes positions lens - new_len .. lens - 1 of every row
  std::vector<int32_t> pos(v.batch);
  for (int b = 0; b < v.batch; ++b) {
    if (lens_host[b] < new_len || lens_host[b] > v.capacity) return OL_ERR_CAPACITY;
    pos[b] = lens_host[b] - new_len;
  }
  if ((st = append_common(v, updated, new_kv, new_len, pos.data(), lens_dev)) != OL_OK) return st;
  if (!valid_page_format(*new_pages)) return OL_ERR_SHAPE;
  const ol_paged_kv k = paged_shape_of(cache);
  if ((st = check_pages(&k, pos.data(), new_len, true, -1)) != OL_OK) return st;
  if ((st = check_hpaged_formats(cache, nullptr, -1, nullptr, pos.data(), new_len)) != OL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // every check of the attention first: an error return means nothing was written
  if ((st = run_attention(OL_LAYOUT_HPAGED, cache, v, q, q_heads, lens_host, lens_dev, new_kv, 0, 1, scale, window,
                          out, out_dtype, workspace, ws_bytes, s, new_len, true)) != OL_OK)
    return st;
  if (fault_injected()) return OL_ERR_INJECTED;
  // the chunk attended uncompressed, then encoded into its pages
  st = run_attention(OL_LAYOUT_HPAGED, cache, v, q, q_heads, lens_host, lens_dev, new_kv, 0, 1, scale, window, out,
                     out_dtype, workspace, ws_bytes, s, new_len);
  if (st != OL_OK) return st;
  AppendParams p = {};
  p.layout = OL_LAYOUT_HPAGED;
  p.dtype = OL_BF16;
  p.batch = v.batch;
  p.kv_heads = v.kv_heads;
  p.head_dim = v.head_dim;
  p.capacity = v.capacity;
  p.new_len = new_len;
  p.values = new_kv;
  p.positions = lens_dev;
  p.positions_are_lens = 1;
  p.pool = cache->pool;
  p.block_table = cache->block_table;
  p.num_pages = cache->num_pages;
  p.page_size = cache->page_size;
  p.max_pages = cache->max_pages;
  p.page_fmt = cache->formats;
  p.new_fmt = *new_pages;
  if (launch_hpaged_append(p, s) != cudaSuccess) return OL_ERR_CUDA;
  // the call's one record: the attention's counts (recorded by run_attention) and the append's
  int64_t appended = 0;
  for (int b = 0; b < v.batch; ++b)
    for (int t = pos[b]; t < pos[b] + new_len; ++t) {
      const ol_page_format& f = hpaged_token_format(cache, b, t, pos[b], *new_pages);
      appended += (int64_t)v.kv_heads *
                  (int64_t)(fmt_row_bytes(f.k.format, v.head_dim) + fmt_row_bytes(f.v.format, v.head_dim));
    }
  for (ol_stats* r : {&t_last, &t_total}) {
    r->storage_append_copied_bytes += appended;
    r->storage_reuse_count += v.batch > 0 ? 2 : 0;
  }
  hpaged_start_pages(cache, pos.data(), new_len, *new_pages);
  return OL_OK;
}

ol_status ol_hpaged_quantize(const ol_hpaged_kv* cache, void* updated, const int32_t* pages_host,
                             const int32_t* pages_dev, const int32_t* valid_host, const int32_t* valid_dev, int32_t n,
                             const ol_page_format* to, ol_stream stream) {
  CacheView v;
  ol_status st = view_hpaged(cache, v);
  if (st != OL_OK) return st;
  if ((st = writable(v, updated)) != OL_OK) return st;
  if (!to) return OL_ERR_NULL;
  if (n < 0) return OL_ERR_SHAPE;
  if (n > 0 && (!pages_host || !pages_dev || !valid_host || !valid_dev)) return OL_ERR_NULL;
  if (!valid_page_format(*to)) return OL_ERR_SHAPE;
  // one head's page rows are staged in shared memory as fp32
  if ((size_t)cache->page_size * cache->head_dim * 4 > 200 * 1024) return OL_ERR_UNSUPPORTED;
  if (n > 0 && (!aligned16(pages_dev) || !aligned16(valid_dev))) return OL_ERR_ALIGN;
  std::vector<char> seen(cache->num_pages, 0);
  for (int i = 0; i < n; ++i) {
    const int page = pages_host[i];
    if (page < 0 || page >= cache->num_pages) return OL_ERR_PAGE;
    if (seen[page]) return OL_ERR_SHAPE;
    seen[page] = 1;
    if (valid_host[i] < 0 || valid_host[i] > cache->page_size) return OL_ERR_CAPACITY;
    if (!valid_page_format(cache->formats_host[page])) return OL_ERR_SHAPE;
  }
  if ((st = no_overlap(v, pages_dev, sizeof(int32_t) * (size_t)n)) != OL_OK) return st;
  if ((st = no_overlap(v, valid_dev, sizeof(int32_t) * (size_t)n)) != OL_OK) return st;
  if ((st = check_owner(v.ranges, v.nranges, v.owner)) != OL_OK) return st;
  {
    // statistics: the converted rows are read in the old formats and written in the new
    ol_stats s = {};
    s.calls = 1;
    const int D = cache->head_dim;
    for (int i = 0; i < n; ++i) {
      const ol_page_format& f = cache->formats_host[pages_host[i]];
      const int64_t rows = (int64_t)valid_host[i] * cache->kv_heads;
      s.kv_payload_bytes_read += rows * (int64_t)(fmt_row_bytes(f.k.format, D) + fmt_row_bytes(f.v.format, D));
      s.dequantized_bytes += rows * D * 4 * ((fmt_affine(f.k.format) ? 1 : 0) + (fmt_affine(f.v.format) ? 1 : 0));
      s.storage_append_copied_bytes += (int64_t)cache->page_size * cache->kv_heads *
                                       (int64_t)(fmt_row_bytes(to->k.format, D) + fmt_row_bytes(to->v.format, D));
    }
    s.storage_reuse_count = n > 0 ? 2 : 0;
    record(s);
  }
  if (fault_injected()) return OL_ERR_INJECTED;
  QuantizeParams p = {};
  p.pool = static_cast<uint8_t*>(cache->pool);
  p.page_fmt = cache->formats;
  p.num_pages = cache->num_pages;
  p.kv_heads = cache->kv_heads;
  p.page_size = cache->page_size;
  p.head_dim = cache->head_dim;
  p.pages = pages_dev;
  p.valid = valid_dev;
  p.n = n;
  p.to = *to;
  if (launch_hpaged_quantize(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return OL_ERR_CUDA;
  for (int i = 0; i < n; ++i) cache->formats_host[pages_host[i]] = *to;
  return OL_OK;
}

}  // extern "C"
