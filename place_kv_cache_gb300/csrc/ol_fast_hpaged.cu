// ol_fast_hpaged.cu -- tensor-core decode attention (and fused append) over
// the heterogeneous paged cache, for head_dim 128, a GQA group of at most 8
// and pages of a multiple of 16 slots: every 16-token tile lies in one page
// and takes that page's K and V formats.
//
// Decomposition as in the bf16 kernel: one CTA per (row, kv head, split),
// warps over 16-token tiles with their own STAGES-deep rings, the shared
// merge. A tile's K and V arrive as the bytes they occupy in the pool: TMA
// 2-D copies of 16 rows through one tensor map per row width (256, 128, 64
// and 32 bytes) whose swizzle keeps the reads below free of bank conflicts.
// FLOAT planes (512-byte rows) are read by the warp from global memory.
//
// Dequantization is exact, inside the MMA operands:
//   S^T = K q^T
//     BFLOAT16: K against bf16 q.  FLOAT: bf16 hi + lo of K against bf16 q.
//     FLOAT16: K against fp16 q * 2^e[col] (e puts the column's largest |q|
//     in [2^14, 2^15), so the conversion of q is exact).
//     Affine codes: the code bits themselves, masked in place, as fp16
//     subnormals c' * 2^(p - 24) (c' = c + 2^(bits-1) for signed formats, so
//     c' >= 0; p the code's bit position in its 16-bit half, at most 8)
//     against the same fp16 q times 2^-p, then
//     s = scale * (2^(24 - e) acc - zp' * sum(q)), zp' the zero point with
//     the same offset. Each code width takes q in its own permuted dimension
//     order: the order in which a lane finds its codes in the tile.
//   O^T += V^T P^T
//     Dense formats: V as stored (FLOAT as bf16 hi + lo) against P^T as
//     bf16 (FLOAT16: fp16) hi + lo.  Affine codes: V^T as the exact fp16
//     difference (1024 + c') - (1024 + zp') against fp16 (P * m)^T hi + lo,
//     where the V scale is m * 2^k (m in [1, 2)): O is held in units of 2^k
//     of the tile's k, rescaled by a power of two when k changes.
//     Every format writes O^T in one permuted dimension order (m-tile 2b + h,
//     row r: dimension 32b + 4r + 2h; row r + 8: the next one), put back in
//     order when the warp state is stored.
// The q operands in their four orders live in shared memory, once per CTA.
// The token being appended takes part uncompressed from new_kv after the tile
// loop; the fused step encodes it into its page in that page's formats.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ol_hpaged.cuh"
#include "ol_merge.cuh"

namespace ol {
namespace {

constexpr int kTok = 16;
constexpr int kRegion = 4096;         // one plane of a tile in a stage: 16 rows of up to 256 bytes
constexpr int kStage = 2 * kRegion;   // K region, V region
constexpr int kHalf = 2048;           // a 16-bit tile's second 64-dimension half
constexpr int kInfo = 8;              // ints of tile information per stage
constexpr float kLazy = 8.f;          // log2 headroom of the lazy softmax maximum

template <int NWARPS, int STAGES, int NG = 1>
struct HpLayout {
  static constexpr int kStages = NWARPS * STAGES * kStage;
  // q operands of each column group: 4 orders x 8 k-steps x 32 lanes x 2 registers
  static constexpr int kQ = NG * 4 * 8 * 32 * 8;
  static constexpr int kQAux = NG * 2 * 8 * 4;  // per column: exponent e and sum of q
  static constexpr int kInfoBytes = NWARPS * STAGES * kInfo * 4;
  static constexpr int kBars = NWARPS * STAGES * 8;
  static constexpr int kMisc = 256 + NWARPS * 8 * 4 * 2 + 8 * 4 * 6 + 2 * 16 * 8 * 4 + 16;
  static constexpr int kTotal = 1024 + kStages + kQ + kQAux + kInfoBytes + kBars + kMisc;
  static constexpr int kBySmem = (228 * 1024) / (kTotal + 1024) > 0 ? (228 * 1024) / (kTotal + 1024) : 1;
  // two column groups take up to 255 registers: one CTA per SM
  static constexpr int kPerSm = NG > 1 ? 1 : (kBySmem < 2 ? kBySmem : 2);
  static_assert(STAGES >= 2, "the merged O lives in warp 0's second stage");
  static_assert(8 * kOStride * 4 <= kStage, "a warp state fits one stage");
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
// FLOAT-page loads in program order (volatile: not hoisted across the MMAs,
// which keeps their registers few)
__device__ __forceinline__ float2 ldg_f2(const float* ptr) {
  float2 v;
  asm volatile("ld.global.nc.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(ptr));
  return v;
}
__device__ __forceinline__ float4 ldg_f4(const float* ptr) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(ptr));
  return v;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) { return __byte_perm(a, b, sel); }
// (a & b) ^ c in one instruction
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hsub2_f16(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// bf16 pair of (x, y) and the pair of their remainders
__device__ __forceinline__ void split_bf16(float x, float y, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(x, y);
  lo = pack_bf16x2(x - __uint_as_float(hi << 16), y - __uint_as_float(hi & 0xffff0000u));
}
__device__ __forceinline__ float2 bc2(float x) { return make_float2(x, x); }
// the same for a packed pair (the remainders by one paired fma: v - hi)
__device__ __forceinline__ void split_bf16(float2 v, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(v.x, v.y);
  const float2 r =
      __ffma2_rn(make_float2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u)), bc2(-1.f), v);
  lo = pack_bf16x2(r.x, r.y);
}
__device__ __forceinline__ void split_f16(float2 v, uint32_t& hi, uint32_t& lo) {
  hi = pack_f16x2(v.x, v.y);
  const float2 r = __ffma2_rn(__half22float2(*reinterpret_cast<__half2*>(&hi)), bc2(-1.f), v);
  lo = pack_f16x2(r.x, r.y);
}

// 2^k as a float: the exponent field directly where it is in range
__device__ __forceinline__ float pow2f(int k) {
  return (k >= -126 && k <= 127) ? __int_as_float((k + 127) << 23) : ldexpf(1.f, k);
}
// floor(log2(x)) of a positive finite x
__device__ __forceinline__ int log2_floor(float x) {
  const int e = (__float_as_int(x) >> 23) & 0xFF;
  return e != 0 ? e - 127 : ilogbf(x);
}

// Bounded wait that lets the warp sleep (suspend-time hint) instead of spinning
// while its tile is in flight; false if the phase did not complete within
// kWaitLimitCycles.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
  return true;
}

// Code offset of a signed format (its codes are read as c + 2^(bits-1)).
__device__ __forceinline__ int code_offset(int f) { return fmt_signed(f) ? 1 << (fmt_bits(f) - 1) : 0; }

// Row of the tensor map of row width fmt_row_bytes(f, 128) that holds
// (page, plane, head g, page slot s).
__device__ __forceinline__ int map_row(const AttnParams& p, int page, int plane, int g, int s, int f) {
  const int per_plane = p.kv_heads * p.page_size * (32 / fmt_bits(f));  // rows of this width per plane
  return (page * 2 + plane) * per_plane + g * p.page_size + s;
}

// -------------------------------------------------------------- the kernel

// CHUNK: a chunked step's attention (grid x = pair of slices of query tokens,
// y = the split): state columns are (query token, head) pairs, each masked to
// its token's window; the history ends where the chunk starts, and the
// chunk's tokens take part uncompressed from new_kv, folded causally into
// warp 0's state after the tile loop. A warp carries two slices' columns (two
// column groups: their own q operands, scores, softmax states and O) and
// decodes each tile's operands once for both. Its own instantiation: the
// decode kernel keeps its own code.
// DUP (a decode step with at most 4 heads per kv head): MMA columns 4..7
// repeat the heads of columns 0..3, so the two halves of P^T (hi and lo)
// travel in one MMA, hi in columns 0..3 and lo in 4..7, added when the state
// is stored. Affine V codes then enter as exact fp16 subnormals c' * 2^-24
// (O in units of 2^(k + 24) on those tiles) and the page's zero point is one
// fp32 sum per column, zp' * sum_t P'[t], subtracted at the end.
template <int NWARPS, int STAGES, bool CHUNK = false, bool DUP = false>
__global__ void __launch_bounds__(NWARPS * 32, HpLayout<NWARPS, STAGES, CHUNK ? 2 : 1>::kPerSm)
    fast_hpaged_kernel(const __grid_constant__ CUtensorMap tm16, const __grid_constant__ CUtensorMap tm8,
                       const __grid_constant__ CUtensorMap tm4, const __grid_constant__ CUtensorMap tm2,
                       const __grid_constant__ AttnParams p) {
  static_assert(!(CHUNK && DUP), "duplicated columns serve a decode step only");
  constexpr int NG = CHUNK ? 2 : 1;  // column groups a warp carries (a chunked step: two slices)
  using L = HpLayout<NWARPS, STAGES, NG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* stages = smem;
  uint2* qsm = reinterpret_cast<uint2*>(smem + L::kStages);            // [group][order][kk][lane]
  int* qexp = reinterpret_cast<int*>(smem + L::kStages + L::kQ);       // [group][8] per column
  float* qsum_h = reinterpret_cast<float*>(qexp + NG * 8);             // [group][8] per column
  uint8_t* after_q = smem + L::kStages + L::kQ + L::kQAux;
  int* info = reinterpret_cast<int*>(after_q);
  uint64_t* bars = reinterpret_cast<uint64_t*>(after_q + L::kInfoBytes);
  Work* sw = reinterpret_cast<Work*>(after_q + L::kInfoBytes + L::kBars);
  float* misc = reinterpret_cast<float*>(after_q + L::kInfoBytes + L::kBars + 256);
  MergeScratch ms;
  ms.wm = misc;
  ms.wl = ms.wm + NWARPS * 8;
  ms.m = ms.wl + NWARPS * 8;
  ms.l = ms.m + 8;
  ms.cm = ms.l + 8;
  ms.cl = ms.cm + 8;
  ms.scr = ms.cl + 8;
  ms.cw = ms.scr + 16;
  ms.wt = ms.cw + 16 * 8;
  ms.flag = reinterpret_cast<int*>(ms.wt + 16 * 8);
  ms.recv_o = ms.recv_m = ms.recv_l = nullptr;  // no cluster

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tm16);
    prefetch_tensormap(&tm8);
    prefetch_tensormap(&tm4);
    prefetch_tensormap(&tm2);
  }
  const uint32_t bar0 = smem_u32(bars + warp * STAGES);
  if (lane == 0) {
    for (int st = 0; st < STAGES; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_mbar_init();
  }
  pdl_wait();
  pdl_launch_dependents();
  // a chunked step's CTA serves NG consecutive slices of query tokens, zs0 .. zs0 + nsl - 1
  const int nslices = CHUNK ? (p.nq + slice_tq(p) - 1) / slice_tq(p) : 1;
  const int zs0 = CHUNK ? NG * query_index(p) : 0;
  const int nsl = CHUNK ? min(NG, nslices - zs0) : 1;
  if (warp == 0) {
    Work w = p.inline_lens ? map_cta_warp(p.lens_inline, p.batch, p.kv_heads, p.capacity, p.window, p.chunk,
                                          cta_index(p), nullptr, 1, p.ordered ? p.row_order : nullptr)
                           : map_cta_warp(p.lens, p.batch, p.kv_heads, p.capacity, p.window, p.chunk, cta_index(p),
                                          p.status);
    if (CHUNK) slice_query(w, p, zs0, zs0 + nsl - 1);
    if (lane == 0) *sw = w;
  }
  __syncthreads();
  const Work w = *sw;
  if (!w.valid) return;

  const int G = p.group;
  // column group g: slice zs0 + g, query tokens gz0[g] .. gzl[g] (a group past the
  // last slice has none: gzl = gz0 - 1); w.hi is one past the last slice's last token
  int gz0[NG], gzl[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    gz0[g] = CHUNK ? slice_first(p, zs0 + g) : 0;
    gzl[g] = CHUNK ? (g < nsl ? gz0[g] + slice_tokens(p, zs0 + g) - 1 : gz0[g] - 1) : 0;
  }
  const int zlast = gzl[nsl - 1];
  const int cur = p.cur_from_new ? w.hi - 1 : -1;
  // history tiles: [t_begin, tend); the current token (a chunk: the chunk's
  // tokens up to the slice's last one, from new_kv) is not read from the cache
  const int hist_end = CHUNK ? w.hi - 1 - zlast : (p.cur_from_new ? w.hi - 1 : w.hi);
  const int tend = min(w.t_end, hist_end);
  const int nsub = tend > w.t_begin ? (tend - w.t_begin + kTok - 1) / kTok : 0;
  const int my_n = nsub > warp ? (nsub - warp + NWARPS - 1) / NWARPS : 0;
  uint8_t* my_stages = stages + warp * STAGES * kStage;
  int* my_info = info + warp * STAGES * kInfo;
  // a chunked step's slices (adjacent in launch order) read the same tiles, the later ones from L2
  const uint64_t pol = CHUNK ? policy_evict_normal() : policy_evict_first();
  const ol_page_format* __restrict__ fmts = p.page_fmt;

  // Look-ahead: lane j holds what the warp needs of its tile la_base + j, so one
  // round of dependent lookups (block table, then format table) serves 32
  // tiles, and the per-tile constants are computed once, 32 tiles at a time:
  //   page, the tile's TMA rows of K and V (-1: a FLOAT plane),
  //   w0 = K format | V format << 4 | (V scale exponent + 256) << 8 | V zero point' << 18,
  //   kbase: S scale (exp2 domain; codes: K scale * 2^24, FLOAT16: 1; times 2^-e per column after),
  //   kbias: K scale * zero point' (exp2 domain; times sum(q) per column after),
  //   mv: the V scale's mantissa in [1, 2) (dense: 1).
  const float sl2 = p.scale_log2;
  int la_base = -64, la_page = 0, la_w0 = 0, la_rowk = 0, la_rowv = 0;
  float la_kbase = 0.f, la_kbias = 0.f, la_mv = 1.f;
  auto look_ahead = [&](int base) {  // whole warp
    la_base = base;
    const int ti = base + lane;
    if (ti < my_n) {
      const int t0 = w.t_begin + (warp + ti * NWARPS) * kTok;
      int page = __ldg(p.block_table + (size_t)w.b * p.max_pages + t0 / p.page_size);
      if (page < 0 || page >= p.num_pages) {
        set_status(p.status, OL_DEVICE_GUARD);
        page = 0;
      }
      const ol_plane_format fk_ = fmts[page].k, fv_ = fmts[page].v;
      const int fk = min(max(fk_.format, 0), (int)OL_FMT_U2), fv = min(max(fv_.format, 0), (int)OL_FMT_U2);
      const int s0 = t0 % p.page_size;
      int kv = 0, vz = 0;
      float mv = 1.f;
      if (fmt_affine(fv)) {
        kv = log2_floor(fv_.scale);
        mv = fv_.scale * pow2f(-kv);
        if (DUP) kv += 24;  // the codes enter as c' * 2^-24
        vz = fv_.zero_point + code_offset(fv);
      }
      la_page = page;
      la_w0 = fk | fv << 4 | (kv + 256) << 8 | vz << 18;
      la_rowk = fk == OL_FMT_F32 ? -1 : map_row(p, page, 0, w.g, s0, fk);
      la_rowv = fv == OL_FMT_F32 ? -1 : map_row(p, page, 1, w.g, s0, fv);
      if (fmt_affine(fk)) {
        la_kbase = fk_.scale * sl2 * 16777216.f;
        la_kbias = fk_.scale * sl2 * (float)(fk_.zero_point + code_offset(fk));
      } else {
        la_kbase = sl2;
        la_kbias = 0.f;
      }
      la_mv = mv;
    }
  };
  // whole warp: tile i's constants from the look-ahead; lane 0 records them
  // for the compute phase and requests the tile's bytes
  auto issue = [&](int i) {
    if (i >= la_base + 32) look_ahead(i);
    const int src = i - la_base;
    const int page = __shfl_sync(0xffffffffu, la_page, src), w0 = __shfl_sync(0xffffffffu, la_w0, src);
    const int rowk = __shfl_sync(0xffffffffu, la_rowk, src), rowv = __shfl_sync(0xffffffffu, la_rowv, src);
    const float kbase = __shfl_sync(0xffffffffu, la_kbase, src), kbias = __shfl_sync(0xffffffffu, la_kbias, src);
    const float mv = __shfl_sync(0xffffffffu, la_mv, src);
    if (lane != 0) return;
    const int st = i % STAGES;
    int* inf = my_info + st * kInfo;
    inf[0] = page;
    inf[1] = w0;
    inf[2] = __float_as_int(kbase);
    inf[3] = __float_as_int(kbias);
    inf[4] = __float_as_int(mv);
    const int fk = w0 & 15, fv = (w0 >> 4) & 15;
    const uint32_t bk = fk == OL_FMT_F32 ? 0u : kTok * (uint32_t)fmt_row_bytes(fk, 128);
    const uint32_t bv = fv == OL_FMT_F32 ? 0u : kTok * (uint32_t)fmt_row_bytes(fv, 128);
    const uint32_t dst = smem_u32(my_stages + st * kStage);
    const uint32_t bar = bar0 + 8 * st;
    fence_proxy_async_smem();  // generic writes to this stage (zeroed rows) before the async-proxy refill
    mbar_arrive_expect_tx(bar, bk + bv);
#pragma unroll
    for (int plane = 0; plane < 2; ++plane) {
      const int row = plane == 0 ? rowk : rowv;
      if (row < 0) continue;
      const uint32_t d = dst + plane * kRegion;
      switch (fmt_bits(plane == 0 ? fk : fv)) {
        case 16:
          tma_load_2d(d, &tm16, 0, row, bar, pol);
          tma_load_2d(d + kHalf, &tm16, 64, row, bar, pol);
          break;
        case 8: tma_load_2d(d, &tm8, 0, row, bar, pol); break;
        case 4: tma_load_2d(d, &tm4, 0, row, bar, pol); break;
        default: tma_load_2d(d, &tm2, 0, row, bar, pol); break;
      }
    }
  };
  for (int i = 0; i < min(my_n, STAGES); ++i) issue(i);

  // ---- q operands of each column group (lane: c = lane % 4, n = lane / 4 =
  // state column: the head, or for a chunked step head n % G of the slice's
  // query token n / G), written once per CTA, group g by warp g
  const int c = lane & 3, n = lane >> 2;
  const int ncol = DUP ? (n & 3) : n;  // the state column of MMA column n
  auto gcols = [&](int g) { return CHUNK ? G * (gzl[g] - gz0[g] + 1) : G; };  // live columns of group g
  // the q row of this lane's column in group g (live: the column exists)
  auto gq = [&](int g, bool& live) -> const uint16_t* {
    live = ncol < gcols(g);
    const int nl = live ? ncol : 0;
    return reinterpret_cast<const uint16_t*>(p.q) +
           (CHUNK ? (((size_t)w.b * p.q_heads + (size_t)w.g * G + nl % G) * p.nq + gz0[g] + nl / G) * 128
                  : ((size_t)w.b * p.q_heads + (size_t)w.g * G + nl) * 128);
  };
  if (warp < NG) {
    const int g = warp;
    bool live;
    const uint16_t* qp = gq(g, live);
    uint2* qg = qsm + g * 4 * 8 * 32;
    // this lane's 32 dims 32c .. 32c + 31 of column n: its exponent e and sum
    uint32_t qraw[16];
    const uint4* src = reinterpret_cast<const uint4*>(qp + 32 * c);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = live ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
      qraw[4 * k] = v.x;
      qraw[4 * k + 1] = v.y;
      qraw[4 * k + 2] = v.z;
      qraw[4 * k + 3] = v.w;
    }
    float qmax = 0.f, qsum = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float lo = __uint_as_float(qraw[k] << 16), hi = __uint_as_float(qraw[k] & 0xffff0000u);
      qmax = fmaxf(qmax, fmaxf(fabsf(lo), fabsf(hi)));
      qsum += lo + hi;
    }
    qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 1));
    qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 2));
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
    const int qe = qmax > 0.f ? 14 - log2_floor(qmax) : 0;  // column n's largest |q| * 2^e in [2^14, 2^15)
    const float s2e_n = pow2f(qe);
    if (c == 0) {
      qexp[g * 8 + n] = qe;
      qsum_h[g * 8 + n] = qsum;
    }
    auto qd = [&](int j) {  // q[n][32c + j] * 2^e as float (j < 32)
      const uint32_t wd = qraw[j >> 1];
      return ((j & 1) ? __uint_as_float(wd & 0xffff0000u) : __uint_as_float(wd << 16)) * s2e_n;
    };
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      // order 0, standard: dims 16kk + 2c, +1 | +8, +9 (bf16 as stored)
      uint2 b;
      b.x = live ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * kk + 2 * c)) : 0u;
      b.y = live ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * kk + 2 * c + 8)) : 0u;
      qg[(0 * 8 + kk) * 32 + lane] = b;
      // order 1, 4-bit codes: kk = 2i + h, e_j = 8i + j: (e_2h, e_2h+4) | (e_2h+1, e_2h+5) / 16
      {
        const int i = kk >> 1, h = kk & 1, e = 8 * i;
        b.x = pack_f16x2(qd(e + 2 * h), qd(e + 2 * h + 4));
        b.y = pack_f16x2(qd(e + 2 * h + 1) * 0.0625f, qd(e + 2 * h + 5) * 0.0625f);
        qg[(1 * 8 + kk) * 32 + lane] = b;
      }
      // order 2, 8-bit codes: d_j = 4kk + j: (d0, d2) | (d1, d3)
      b.x = pack_f16x2(qd(4 * kk), qd(4 * kk + 2));
      b.y = pack_f16x2(qd(4 * kk + 1), qd(4 * kk + 3));
      qg[(2 * 8 + kk) * 32 + lane] = b;
      // order 3, 2-bit codes: word w = kk / 4, pairs j = 2(kk % 4) (+1): (16w + j, 16w + j + 8) / 4^f(j),
      // f(j) = j below 5, j - 5 from 5 (the bit position / 2 of the masked code)
      {
        const int wv = kk >> 2, j0 = 2 * (kk & 3), j1 = j0 + 1;
        const float f0 = pow2f(-2 * (j0 < 5 ? j0 : j0 - 5)), f1 = pow2f(-2 * (j1 < 5 ? j1 : j1 - 5));
        b.x = pack_f16x2(qd(16 * wv + j0) * f0, qd(16 * wv + j0 + 8) * f0);
        b.y = pack_f16x2(qd(16 * wv + j1) * f1, qd(16 * wv + j1 + 8) * f1);
        qg[(3 * 8 + kk) * 32 + lane] = b;
      }
    }
  }
  __syncthreads();
  // per group: 2^e of this lane's B-operand column n; 2^-e and sum(q) of its
  // state columns 2c, 2c + 1
  float s2e[NG], qs0[NG], qs1[NG], pne0[NG], pne1[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    s2e[g] = pow2f(qexp[g * 8 + n]);
    qs0[g] = qsum_h[g * 8 + 2 * c];
    qs1[g] = qsum_h[g * 8 + 2 * c + 1];
    pne0[g] = pow2f(-qexp[g * 8 + 2 * c]);
    pne1[g] = pow2f(-qexp[g * 8 + 2 * c + 1]);
  }
  const uint32_t qbase = smem_u32(qsm) + lane * 8;
  auto qop = [&](int order, int kk, int g) { return lds_v2(qbase + ((g * 4 + order) * 8 + kk) * 256); };

  // visible history of this lane's state columns 2c, 2c + 1 of each group: a
  // chunked step's column from its own query token's window start
  int clo0[NG], clo1[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    clo0[g] = clo1[g] = w.lo;
    if (CHUNK && p.window_q >= 0) {
      const int t0c = min((2 * c) / G, gzl[g] - gz0[g]), t1c = min((2 * c + 1) / G, gzl[g] - gz0[g]);
      clo0[g] = max(w.lo, hist_end + gz0[g] + t0c - p.window_q);
      clo1[g] = max(w.lo, hist_end + gz0[g] + t1c - p.window_q);
    }
  }

  float o[NG][8][4];
  float mr[NG][2], lr[NG][2];  // running maximum and sum of the lane's columns 2c, 2c + 1 of each group
#pragma unroll
  for (int g = 0; g < NG; ++g) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[g][mt][0] = o[g][mt][1] = o[g][mt][2] = o[g][mt][3] = 0.f;
    mr[g][0] = mr[g][1] = -INFINITY;
    lr[g][0] = lr[g][1] = 0.f;
  }
  int ko = 0;  // O is held in units of 2^ko
  // DUP: the zero-point term of the lane's columns 2c, 2c + 1 over its tokens
  // (units of O times 2^24), and 1 on the lanes of columns 4..7 (the lo half)
  float zc0 = 0.f, zc1 = 0.f;
  const float hsel = DUP && c >= 2 ? 1.f : 0.f;

  const int mi = lane >> 3, r8 = lane & 7;
  const int rK = r8 + 8 * (mi & 1), cK = mi >> 1;  // ldmatrix roles for 16-bit K
  const uint8_t* pool = reinterpret_cast<const uint8_t*>(p.pool);
  const size_t slot_bytes = (size_t)p.kv_heads * p.page_size * 128 * 8;  // 2 planes x 128 dims x 4 bytes

  for (int i = 0; i < my_n; ++i) {
    const int st = i % STAGES;
    if (!mbar_wait_sleep(bar0 + 8 * st, (i / STAGES) & 1)) {
      if (lane == 0) set_status(p.status, OL_DEVICE_GUARD);
      break;
    }
    const int t0 = w.t_begin + (warp + i * NWARPS) * kTok;
    const int* inf = my_info + st * kInfo;
    const int w0 = inf[1];
    const int fk = w0 & 15, fv = (w0 >> 4) & 15, kv = ((w0 >> 8) & 1023) - 256, vz = w0 >> 18;
    const float kbase = __int_as_float(inf[2]), kbias = __int_as_float(inf[3]), mv = __int_as_float(inf[4]);
    const uint32_t sK = smem_u32(my_stages + st * kStage), sV = sK + kRegion;
    // a FLOAT plane's rows in global memory (page slot s0 of head g)
    auto gplane = [&](int plane) {
      return pool + (size_t)inf[0] * slot_bytes + (size_t)plane * (slot_bytes / 2) +
             ((size_t)w.g * p.page_size + t0 % p.page_size) * 512;
    };

    // V rows at or past the history end hold no data: zero their bytes
    const int vhi = hist_end - t0;
    if (vhi < kTok && fv != OL_FMT_F32) {
      const int rb = (int)fmt_row_bytes(fv, 128), cpr = rb / 16;
      uint8_t* v = my_stages + st * kStage + kRegion;
      for (int idx = lane; idx < (kTok - vhi) * cpr; idx += 32) {
        const int r = vhi + idx / cpr, ch = idx % cpr;
        const int off = rb == 256 ? (ch >> 3) * kHalf + r * 128 + (ch & 7) * 16 : r * rb + ch * 16;
        *reinterpret_cast<uint4*>(v + off) = make_uint4(0, 0, 0, 0);
      }
    }
    __syncwarp();

    // ---- S^T = K q^T, even and odd k-steps in two accumulators (shorter MMA
    // chains), one pair per column group; a tile's K operands serve every group
    float sa[NG][4], sb[NG][4];
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int j = 0; j < 4; ++j) sa[g][j] = sb[g][j] = 0.f;
    if (fk == OL_FMT_BF16 || fk == OL_FMT_F16) {
      const bool h16 = fk == OL_FMT_F16;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int ch = 2 * kk + cK;
        uint32_t a0, a1, a2, a3;
        ldsm_x4(sK + (ch >> 3) * kHalf + rK * 128 + (((ch & 7) ^ r8) << 4), a0, a1, a2, a3);
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const uint2 q = qop(0, kk, g);
          float(&acc)[4] = (kk & 1) ? sb[g] : sa[g];
          if (h16) {
            const float e = s2e[g];
            const uint32_t b0 = pack_f16x2(__uint_as_float(q.x << 16) * e, __uint_as_float(q.x & 0xffff0000u) * e);
            const uint32_t b1 = pack_f16x2(__uint_as_float(q.y << 16) * e, __uint_as_float(q.y & 0xffff0000u) * e);
            mma_f16_16816(acc, a0, a1, a2, a3, b0, b1);
          } else {
            mma_bf16_16816(acc, a0, a1, a2, a3, q.x, q.y);
          }
        }
      }
    } else if (fk == OL_FMT_F32) {
      const uint8_t* gK = gplane(0);
      const float* ra = reinterpret_cast<const float*>(gK + (size_t)n * 512);
      const float* rb = reinterpret_cast<const float*>(gK + (size_t)(n + 8) * 512);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int d = 16 * kk + 2 * c;
        const float2 x0 = ldg_f2(ra + d), x1 = ldg_f2(rb + d);
        const float2 x2 = ldg_f2(ra + d + 8), x3 = ldg_f2(rb + d + 8);
        uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
        split_bf16(x0.x, x0.y, h0, l0);
        split_bf16(x1.x, x1.y, h1, l1);
        split_bf16(x2.x, x2.y, h2, l2);
        split_bf16(x3.x, x3.y, h3, l3);
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const uint2 q = qop(0, kk, g);
          mma_bf16_16816(sa[g], h0, h1, h2, h3, q.x, q.y);
          mma_bf16_16816(sb[g], l0, l1, l2, l3, q.x, q.y);
        }
      }
    } else {
      // affine codes: A = the code bits masked in place (fp16 subnormals), in the width's q order
      const int bits = fmt_bits(fk);
      const bool sgn = fmt_signed(fk);
      if (bits == 8) {
        // rows n and n + 8: this lane's 32 bytes (dims 32c .. 32c + 31) as 8 words of 4 dims
        uint32_t ya[8], yb[8];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint4 va = lds_v4(sK + n * 128 + (((2 * c + m) ^ (n & 7)) << 4));
          const uint4 vb = lds_v4(sK + (n + 8) * 128 + (((2 * c + m) ^ (n & 7)) << 4));
          ya[4 * m] = va.x; ya[4 * m + 1] = va.y; ya[4 * m + 2] = va.z; ya[4 * m + 3] = va.w;
          yb[4 * m] = vb.x; yb[4 * m + 1] = vb.y; yb[4 * m + 2] = vb.z; yb[4 * m + 3] = vb.w;
        }
        // the offset-binary flip of signed codes inside the mask: (x ^ f) & m = (x & m) ^ (f & m)
        const uint32_t fm = sgn ? 0x00800080u : 0u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t x = ya[kk], y = yb[kk];
          const uint32_t a0 = and_xor(x, 0x00FF00FFu, fm), a1 = and_xor(y, 0x00FF00FFu, fm);
          const uint32_t a2 = and_xor(x >> 8, 0x00FF00FFu, fm), a3 = and_xor(y >> 8, 0x00FF00FFu, fm);
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            const uint2 q = qop(2, kk, g);
            mma_f16_16816((kk & 1) ? sb[g] : sa[g], a0, a1, a2, a3, q.x, q.y);
          }
        }
      } else if (bits == 4) {
        const int sw = (n >> 1) & 3;  // rows n and n + 8 share the 64-byte swizzle phase
        const uint4 va = lds_v4(sK + n * 64 + ((c ^ sw) << 4));
        const uint4 vb = lds_v4(sK + (n + 8) * 64 + ((c ^ sw) << 4));
        // the flip of signed codes inside the masks, as for 8 bits
        const uint32_t fl = sgn ? 0x00080008u : 0u, fh = sgn ? 0x00800080u : 0u;
        const uint32_t xa[4] = {va.x, va.y, va.z, va.w}, xb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
          // nibbles j = 0, 4 | 1, 5 (x16) in place; then 2, 6 | 3, 7 (x16) after a shift by 8
          const uint32_t ta = xa[ii] >> 8, tb = xb[ii] >> 8;
          const uint32_t a0 = and_xor(xa[ii], 0x000F000Fu, fl), a1 = and_xor(xb[ii], 0x000F000Fu, fl);
          const uint32_t a2 = and_xor(xa[ii], 0x00F000F0u, fh), a3 = and_xor(xb[ii], 0x00F000F0u, fh);
          const uint32_t c0 = and_xor(ta, 0x000F000Fu, fl), c1 = and_xor(tb, 0x000F000Fu, fl);
          const uint32_t c2 = and_xor(ta, 0x00F000F0u, fh), c3 = and_xor(tb, 0x00F000F0u, fh);
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            const uint2 q0 = qop(1, 2 * ii, g), q1 = qop(1, 2 * ii + 1, g);
            mma_f16_16816(sa[g], a0, a1, a2, a3, q0.x, q0.y);
            mma_f16_16816(sb[g], c0, c1, c2, c3, q1.x, q1.y);
          }
        }
      } else {
        const int sw = (n >> 2) & 1;  // rows n and n + 8 share the 32-byte swizzle phase
        const uint2 va = lds_v2(sK + n * 32 + (((c >> 1) ^ sw) << 4) + 8 * (c & 1));
        const uint2 vb = lds_v2(sK + (n + 8) * 32 + (((c >> 1) ^ sw) << 4) + 8 * (c & 1));
        // the flip of signed codes inside the masks, as for 8 bits (0xAA.. >> 10 keeps its
        // pattern on the masked bits)
        const uint32_t flip = sgn ? 0xAAAAAAAAu : 0u;
        const uint32_t za[2] = {va.x, va.y}, zb[2] = {vb.x, vb.y};
#pragma unroll
        for (int wv = 0; wv < 2; ++wv) {
          // code pairs (j, j + 8) of the word: j < 5 masked in place (bit 2j), j >= 5 after a shift by 10
          const uint32_t ta = za[wv] >> 10, tb = zb[wv] >> 10;
#pragma unroll
          for (int k2 = 0; k2 < 4; ++k2) {
            const int j0 = 2 * k2, j1 = j0 + 1;
            const uint32_t m0 = 0x00030003u << (2 * (j0 < 5 ? j0 : j0 - 5));
            const uint32_t m1 = 0x00030003u << (2 * (j1 < 5 ? j1 : j1 - 5));
            const uint32_t a0 = and_xor(j0 < 5 ? za[wv] : ta, m0, flip & m0);
            const uint32_t a1 = and_xor(j0 < 5 ? zb[wv] : tb, m0, flip & m0);
            const uint32_t a2 = and_xor(j1 < 5 ? za[wv] : ta, m1, flip & m1);
            const uint32_t a3 = and_xor(j1 < 5 ? zb[wv] : tb, m1, flip & m1);
#pragma unroll
            for (int g = 0; g < NG; ++g) {
              const uint2 q = qop(3, 4 * wv + k2, g);
              mma_f16_16816((k2 & 1) ? sb[g] : sa[g], a0, a1, a2, a3, q.x, q.y);
            }
          }
        }
      }
    }

    // ---- online softmax on the S^T columns (exp2 domain), lazy maximum: the
    // running maximum moves only when a score passes it by more than kLazy, so
    // most tiles skip the warp reduction and the rescale (weights stay <= 2^kLazy)
    const int ta_ = t0 + n, tb_ = ta_ + 8;
    const bool va_ = ta_ < tend, vb_ = tb_ < tend;
    // S scale per column: kbase, times 2^-e for fp16-q formats; codes subtract kbias * sum(q)
    const bool kq16 = fk != OL_FMT_BF16 && fk != OL_FMT_F32;
    float pw[NG][4];  // weights: (token n, column 2c), (n, 2c + 1), (n + 8, 2c), (n + 8, 2c + 1)
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      float s00, s01, s10, s11;
      if constexpr (CHUNK) {  // columns (2c, 2c + 1) as packed pairs (measured: faster for chunks only)
        const float2 km = kq16 ? __fmul2_rn(bc2(kbase), make_float2(pne0[g], pne1[g])) : bc2(kbase);
        const float2 kbn = __fmul2_rn(bc2(-kbias), make_float2(qs0[g], qs1[g]));
        const float2 ra =
            __ffma2_rn(__fadd2_rn(make_float2(sa[g][0], sa[g][1]), make_float2(sb[g][0], sb[g][1])), km, kbn);
        const float2 rb =
            __ffma2_rn(__fadd2_rn(make_float2(sa[g][2], sa[g][3]), make_float2(sb[g][2], sb[g][3])), km, kbn);
        s00 = va_ && ta_ >= clo0[g] ? ra.x : -INFINITY;
        s01 = va_ && ta_ >= clo1[g] ? ra.y : -INFINITY;
        s10 = vb_ && tb_ >= clo0[g] ? rb.x : -INFINITY;
        s11 = vb_ && tb_ >= clo1[g] ? rb.y : -INFINITY;
      } else {
        const float kmul0 = kq16 ? kbase * pne0[g] : kbase, kmul1 = kq16 ? kbase * pne1[g] : kbase;
        const float kb0 = kbias * qs0[g], kb1 = kbias * qs1[g];
        s00 = va_ && ta_ >= clo0[g] ? fmaf(sa[g][0] + sb[g][0], kmul0, -kb0) : -INFINITY;
        s01 = va_ && ta_ >= clo1[g] ? fmaf(sa[g][1] + sb[g][1], kmul1, -kb1) : -INFINITY;
        s10 = vb_ && tb_ >= clo0[g] ? fmaf(sa[g][2] + sb[g][2], kmul0, -kb0) : -INFINITY;
        s11 = vb_ && tb_ >= clo1[g] ? fmaf(sa[g][3] + sb[g][3], kmul1, -kb1) : -INFINITY;
      }
      if (__any_sync(0xffffffffu, fmaxf(s00, s10) > mr[g][0] + kLazy || fmaxf(s01, s11) > mr[g][1] + kLazy)) {
        float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(mr[g][0], mx0), mn1 = fmaxf(mr[g][1], mx1);
        const float b0 = mn0 == -INFINITY ? 0.f : mn0, b1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = fast_exp2(mr[g][0] - b0), al1 = fast_exp2(mr[g][1] - b1);
        lr[g][0] *= al0;
        lr[g][1] *= al1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[g][mt][0] *= al0;
          o[g][mt][1] *= al1;
          o[g][mt][2] *= al0;
          o[g][mt][3] *= al1;
        }
        if constexpr (DUP) {
          zc0 *= al0;
          zc1 *= al1;
        }
        mr[g][0] = mn0;
        mr[g][1] = mn1;
      }
      const float b0 = mr[g][0] == -INFINITY ? 0.f : mr[g][0], b1 = mr[g][1] == -INFINITY ? 0.f : mr[g][1];
      pw[g][0] = fast_exp2(s00 - b0);
      pw[g][1] = fast_exp2(s01 - b1);
      pw[g][2] = fast_exp2(s10 - b0);
      pw[g][3] = fast_exp2(s11 - b1);
      lr[g][0] += pw[g][0] + pw[g][2];
      lr[g][1] += pw[g][1] + pw[g][3];
    }
    // O is held in units of 2^kv of the tile's V scale exponent (dense: 0)
    if (kv != ko) {
      const float f = pow2f(ko - kv);
#pragma unroll
      for (int g = 0; g < NG; ++g)
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int j = 0; j < 4; ++j) o[g][mt][j] *= f;
      if constexpr (DUP) {
        zc0 *= f;
        zc1 *= f;
      }
      ko = kv;
    }

    // ---- O^T += V^T P^T (dimension order: m-tile 2bb + hh, row n -> 32bb + 4n + 2hh, row n + 8 -> + 1)
    const int TA = 2 * c, TB = 2 * c + 1, TC = 2 * c + 8, TD = 2 * c + 9;  // this lane's tokens (k rows)
    const bool half_p = fv != OL_FMT_BF16 && fv != OL_FMT_F32;  // P^T in fp16 (else bf16)
    uint32_t ph0[NG], ph1[NG], pl0[NG], pl1[NG];  // per group: P^T hi and lo (DUP: hi | lo in ph)
    if constexpr (DUP) {
      // hi on the lanes of columns 0..3, lo = what hi leaves on those of 4..7
      const float p00 = pw[0][0], p01 = pw[0][1], p10 = pw[0][2], p11 = pw[0][3];
      pl0[0] = pl1[0] = 0u;
      if (half_p) {
        const float x0 = p00 * mv, x1 = p01 * mv, x2 = p10 * mv, x3 = p11 * mv;
        uint32_t h0 = pack_f16x2(x0, x1), h1 = pack_f16x2(x2, x3);
        const float2 f0 = __half22float2(*reinterpret_cast<__half2*>(&h0));
        const float2 f1 = __half22float2(*reinterpret_cast<__half2*>(&h1));
        ph0[0] = movmatrix_trans(pack_f16x2(fmaf(-hsel, f0.x, x0), fmaf(-hsel, f0.y, x1)));
        ph1[0] = movmatrix_trans(pack_f16x2(fmaf(-hsel, f1.x, x2), fmaf(-hsel, f1.y, x3)));
        if (fmt_affine(fv)) {  // the page's zero point, times the weights as they are
          const float z = (float)vz;
          zc0 = fmaf(z, x0 + x2, zc0);
          zc1 = fmaf(z, x1 + x3, zc1);
        }
      } else {
        const uint32_t h0 = pack_bf16x2(p00, p01), h1 = pack_bf16x2(p10, p11);
        ph0[0] = movmatrix_trans(pack_bf16x2(fmaf(-hsel, __uint_as_float(h0 << 16), p00),
                                             fmaf(-hsel, __uint_as_float(h0 & 0xffff0000u), p01)));
        ph1[0] = movmatrix_trans(pack_bf16x2(fmaf(-hsel, __uint_as_float(h1 << 16), p10),
                                             fmaf(-hsel, __uint_as_float(h1 & 0xffff0000u), p11)));
      }
    } else {
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        uint32_t h0, l0, h1, l1;
        if (half_p) {
          split_f16(__fmul2_rn(make_float2(pw[g][0], pw[g][1]), bc2(mv)), h0, l0);
          split_f16(__fmul2_rn(make_float2(pw[g][2], pw[g][3]), bc2(mv)), h1, l1);
        } else {
          split_bf16(make_float2(pw[g][0], pw[g][1]), h0, l0);
          split_bf16(make_float2(pw[g][2], pw[g][3]), h1, l1);
        }
        ph0[g] = movmatrix_trans(h0);
        ph1[g] = movmatrix_trans(h1);
        pl0[g] = movmatrix_trans(l0);
        pl1[g] = movmatrix_trans(l1);
      }
    }
    if (fv == OL_FMT_F32) {
      // V from global memory; rows at or past the history end count as zero
      const uint8_t* gV = gplane(1);
      const int vrow[4] = {TA, TB, TC, TD};
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        float4 x[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          x[k] = ldg_f4(reinterpret_cast<const float*>(gV + (size_t)vrow[k] * 512) + 32 * bb + 4 * n);
          if (vrow[k] >= vhi) x[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float xa0 = hh ? x[0].z : x[0].x, xa1 = hh ? x[0].w : x[0].y;
          const float xb0 = hh ? x[1].z : x[1].x, xb1 = hh ? x[1].w : x[1].y;
          const float xc0 = hh ? x[2].z : x[2].x, xc1 = hh ? x[2].w : x[2].y;
          const float xd0 = hh ? x[3].z : x[3].x, xd1 = hh ? x[3].w : x[3].y;
          uint32_t a0h, a0l, a1h, a1l, a2h, a2l, a3h, a3l;
          split_bf16(xa0, xb0, a0h, a0l);
          split_bf16(xa1, xb1, a1h, a1l);
          split_bf16(xc0, xd0, a2h, a2l);
          split_bf16(xc1, xd1, a3h, a3l);
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            mma_bf16_16816(o[g][2 * bb + hh], a0h, a1h, a2h, a3h, ph0[g], ph1[g]);
            if (!DUP) mma_bf16_16816(o[g][2 * bb + hh], a0h, a1h, a2h, a3h, pl0[g], pl1[g]);
            mma_bf16_16816(o[g][2 * bb + hh], a0l, a1l, a2l, a3l, ph0[g], ph1[g]);
          }
        }
      }
    } else if (fv == OL_FMT_BF16 || fv == OL_FMT_F16) {
      const bool h16 = fv == OL_FMT_F16;
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        // 8 bytes (dims 32bb + 4n .. + 3) of each of the four token rows
        const int e = 32 * (bb & 1) + 4 * n;  // element within the 64-dim half
        const int ch = e >> 3, sub = (e & 7) * 2;
        const uint32_t hb = sV + (bb >> 1) * kHalf + sub;
        const uint2 wa = lds_v2(hb + TA * 128 + ((ch ^ (TA & 7)) << 4));
        const uint2 wb = lds_v2(hb + TB * 128 + ((ch ^ (TB & 7)) << 4));
        const uint2 wc = lds_v2(hb + TC * 128 + ((ch ^ (TC & 7)) << 4));
        const uint2 wd = lds_v2(hb + TD * 128 + ((ch ^ (TD & 7)) << 4));
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t xa = hh ? wa.y : wa.x, xb = hh ? wb.y : wb.x;
          const uint32_t xc = hh ? wc.y : wc.x, xd = hh ? wd.y : wd.x;
          const uint32_t a0 = prmt(xa, xb, 0x5410u), a1 = prmt(xa, xb, 0x7632u);
          const uint32_t a2 = prmt(xc, xd, 0x5410u), a3 = prmt(xc, xd, 0x7632u);
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            if (h16) {
              mma_f16_16816(o[g][2 * bb + hh], a0, a1, a2, a3, ph0[g], ph1[g]);
              if (!DUP) mma_f16_16816(o[g][2 * bb + hh], a0, a1, a2, a3, pl0[g], pl1[g]);
            } else {
              mma_bf16_16816(o[g][2 * bb + hh], a0, a1, a2, a3, ph0[g], ph1[g]);
              if (!DUP) mma_bf16_16816(o[g][2 * bb + hh], a0, a1, a2, a3, pl0[g], pl1[g]);
            }
          }
        }
      }
    } else {
      // affine codes: V^T as exact fp16 (1024 + c') - (1024 + zp') against (P * m)^T
      const int bits = fmt_bits(fv);
      const bool sgn = fmt_signed(fv);
      const uint32_t zf = (uint32_t)__half_as_ushort(__int2half_rn(1024 + vz));
      const uint32_t zpair = zf | (zf << 16);
      auto add_tile = [&](int mt, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
        if constexpr (DUP) {  // c' * 2^-24 as they are; the zero point is in zc
          mma_f16_16816(o[0][mt], a0, a1, a2, a3, ph0[0], ph1[0]);
          return;
        }
        a0 = hsub2_f16(a0, zpair);
        a1 = hsub2_f16(a1, zpair);
        a2 = hsub2_f16(a2, zpair);
        a3 = hsub2_f16(a3, zpair);
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          mma_f16_16816(o[g][mt], a0, a1, a2, a3, ph0[g], ph1[g]);
          mma_f16_16816(o[g][mt], a0, a1, a2, a3, pl0[g], pl1[g]);
        }
      };
      // the offset-binary flip of signed codes, and (not DUP) the fp16 1024 around them
      const uint32_t hi1024 = DUP ? 0u : 0x64006400u;
      if (bits == 8) {
        const uint32_t magic = (sgn ? 0x00800080u : 0u) | hi1024;
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          const int ch = 2 * bb + (n >> 2), sub = 4 * (n & 3);
          const uint32_t xa = lds_u32(sV + TA * 128 + ((ch ^ (TA & 7)) << 4) + sub);
          const uint32_t xb = lds_u32(sV + TB * 128 + ((ch ^ (TB & 7)) << 4) + sub);
          const uint32_t xc = lds_u32(sV + TC * 128 + ((ch ^ (TC & 7)) << 4) + sub);
          const uint32_t xd = lds_u32(sV + TD * 128 + ((ch ^ (TD & 7)) << 4) + sub);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint32_t s0_ = (2 * hh) | ((4 + 2 * hh) << 8), s1_ = (2 * hh + 1) | ((5 + 2 * hh) << 8);
            add_tile(2 * bb + hh, and_xor(prmt(xa, xb, s0_), 0x00FF00FFu, magic),
                     and_xor(prmt(xa, xb, s1_), 0x00FF00FFu, magic), and_xor(prmt(xc, xd, s0_), 0x00FF00FFu, magic),
                     and_xor(prmt(xc, xd, s1_), 0x00FF00FFu, magic));
          }
        }
      } else if (bits == 4) {
        const uint32_t magic = (sgn ? 0x00080008u : 0u) | hi1024;
#pragma unroll
        for (int bp = 0; bp < 2; ++bp) {
          // matrices (tokens 0-7 | 8-15) x (32-dim blocks 2bp | 2bp + 1)
          const int t = r8 + 8 * (mi & 1), cb = 2 * bp + (mi >> 1);
          uint32_t r0, r1, r2, r3;
          ldsm_x4_trans(sV + t * 64 + ((cb ^ ((t >> 1) & 3)) << 4), r0, r1, r2, r3);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint32_t x01 = q ? r2 : r0, x89 = q ? r3 : r1;  // tokens 2c, 2c+1 | 2c+8, 2c+9
            const int bb = 2 * bp + q;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
              add_tile(2 * bb + hh, and_xor(x01 >> (8 * hh), 0x000F000Fu, magic),
                       and_xor(x01 >> (8 * hh + 4), 0x000F000Fu, magic),
                       and_xor(x89 >> (8 * hh), 0x000F000Fu, magic),
                       and_xor(x89 >> (8 * hh + 4), 0x000F000Fu, magic));
          }
        }
      } else {
        const uint32_t magic = (sgn ? 0x00020002u : 0u) | hi1024;
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          // byte 8bb + n of each token row: dims 32bb + 4n .. + 3
          const int x = 8 * bb + n, ch = x >> 4, sub = x & 15;
          const uint32_t ba = lds_u8(sV + TA * 32 + ((ch ^ ((TA >> 2) & 1)) << 4) + sub);
          const uint32_t bbv = lds_u8(sV + TB * 32 + ((ch ^ ((TB >> 2) & 1)) << 4) + sub);
          const uint32_t bc = lds_u8(sV + TC * 32 + ((ch ^ ((TC >> 2) & 1)) << 4) + sub);
          const uint32_t bd = lds_u8(sV + TD * 32 + ((ch ^ ((TD >> 2) & 1)) << 4) + sub);
          const uint32_t xab = prmt(ba, bbv, 0x1410u), xcd = prmt(bc, bd, 0x1410u);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            add_tile(2 * bb + hh, and_xor(xab >> (4 * hh), 0x00030003u, magic),
                     and_xor(xab >> (4 * hh + 2), 0x00030003u, magic), and_xor(xcd >> (4 * hh), 0x00030003u, magic),
                     and_xor(xcd >> (4 * hh + 2), 0x00030003u, magic));
        }
      }
    }
    __syncwarp();
    if (i + STAGES < my_n) issue(i + STAGES);
    __syncwarp();
  }

  if constexpr (DUP) {
    // the zero-point term, summed over the tile rows (lanes n), off every dim
    // on the hi lanes (units of O: 2^-24); then the lo columns added in
    float z0s = zc0, z1s = zc1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      z0s += __shfl_xor_sync(0xffffffffu, z0s, off);
      z1s += __shfl_xor_sync(0xffffffffu, z1s, off);
    }
    z0s = c < 2 ? z0s * 5.9604644775390625e-8f : 0.f;
    z1s = c < 2 ? z1s * 5.9604644775390625e-8f : 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      o[0][mt][0] -= z0s;
      o[0][mt][1] -= z1s;
      o[0][mt][2] -= z0s;
      o[0][mt][3] -= z1s;
#pragma unroll
      for (int j = 0; j < 4; ++j) o[0][mt][j] += __shfl_xor_sync(0xffffffffu, o[0][mt][j], 2);
    }
  }
  if (ko != 0) {
    const float f = pow2f(ko);
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) o[g][mt][j] *= f;
  }

  // ---- the current token, uncompressed from new_kv, in warp 0's state; the
  // fused step also encodes it into its page
  if (cur >= w.t_begin && cur < w.t_end && cur >= 0) {
    const uint16_t* nk = reinterpret_cast<const uint16_t*>(p.new_kv) + ((size_t)w.b * p.kv_heads + w.g) * 128;
    const uint16_t* nv = reinterpret_cast<const uint16_t*>(p.new_kv) +
                         (((size_t)p.batch + w.b) * p.kv_heads + w.g) * 128;
    if (warp == 0 && CHUNK) {
      // group g: the chunk's tokens 0 .. gzl[g], uncompressed: token t is
      // visible to column j (query token zj = gz0[g] + j / G) if t <= zj and,
      // with a window, t >= zj - window
      const size_t kv_row = ((size_t)w.b * p.kv_heads + w.g) * p.nq;
      const uint16_t* ck = reinterpret_cast<const uint16_t*>(p.new_kv) + kv_row * 128;
      const uint16_t* cv = reinterpret_cast<const uint16_t*>(p.new_kv) +
                           ((size_t)p.batch * p.kv_heads * p.nq + kv_row) * 128;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        if (g >= nsl) break;
        bool live;
        const uint16_t* qp = gq(g, live);
        const int ncols = gcols(g);
        const int zc0 = gz0[g] + (2 * c) / G, zc1 = gz0[g] + (2 * c + 1) / G;
        for (int t = 0; t <= gzl[g]; ++t) {
          const uint16_t* kt = ck + (size_t)t * 128;
          const uint16_t* vt = cv + (size_t)t * 128;
          float part = 0.f;
          if (live) {
#pragma unroll 8
            for (int d = 32 * c; d < 32 * c + 32; ++d)
              part = fmaf(bf16_bits_to_float(qp[d]), bf16_bits_to_float(kt[d]), part);
          }
          part += __shfl_xor_sync(0xffffffffu, part, 1);
          part += __shfl_xor_sync(0xffffffffu, part, 2);
          const float sc0 = __shfl_sync(0xffffffffu, part, 8 * c) * sl2;
          const float sc1 = __shfl_sync(0xffffffffu, part, 8 * c + 4) * sl2;
          const bool v0 = 2 * c < ncols && t <= zc0 && (p.window_q < 0 || t >= zc0 - p.window_q);
          const bool v1 = 2 * c + 1 < ncols && t <= zc1 && (p.window_q < 0 || t >= zc1 - p.window_q);
          const float s0c = v0 ? sc0 : -INFINITY, s1c = v1 ? sc1 : -INFINITY;
          const float mn0 = fmaxf(mr[g][0], s0c), mn1 = fmaxf(mr[g][1], s1c);
          const float b0 = mn0 == -INFINITY ? 0.f : mn0, b1 = mn1 == -INFINITY ? 0.f : mn1;
          const float al0 = fast_exp2(mr[g][0] - b0), al1 = fast_exp2(mr[g][1] - b1);
          const float pc0 = fast_exp2(s0c - b0), pc1 = fast_exp2(s1c - b1);
          lr[g][0] = lr[g][0] * al0 + (n == 0 ? pc0 : 0.f);
          lr[g][1] = lr[g][1] * al1 + (n == 0 ? pc1 : 0.f);
          mr[g][0] = mn0;
          mr[g][1] = mn1;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const int da = 32 * (mt >> 1) + 4 * n + 2 * (mt & 1);
            const float va = bf16_bits_to_float(vt[da]), vb = bf16_bits_to_float(vt[da + 1]);
            o[g][mt][0] = fmaf(pc0, va, o[g][mt][0] * al0);
            o[g][mt][1] = fmaf(pc1, va, o[g][mt][1] * al1);
            o[g][mt][2] = fmaf(pc0, vb, o[g][mt][2] * al0);
            o[g][mt][3] = fmaf(pc1, vb, o[g][mt][3] * al1);
          }
        }
      }
    } else if (warp == 0) {
      bool live;
      const uint16_t* qp = gq(0, live);
      float part = 0.f;
      if (live) {
#pragma unroll 8
        for (int d = 32 * c; d < 32 * c + 32; ++d) part = fmaf(bf16_bits_to_float(qp[d]), bf16_bits_to_float(nk[d]), part);
      }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      // head n's score sits in lanes 4n .. 4n + 3; this lane's columns are 2c, 2c + 1
      const float sc0 = __shfl_sync(0xffffffffu, part, 8 * c) * sl2;
      const float sc1 = __shfl_sync(0xffffffffu, part, 8 * c + 4) * sl2;
      const float s0c = 2 * c < G ? sc0 : -INFINITY, s1c = 2 * c + 1 < G ? sc1 : -INFINITY;
      const float mn0 = fmaxf(mr[0][0], s0c), mn1 = fmaxf(mr[0][1], s1c);
      const float b0 = mn0 == -INFINITY ? 0.f : mn0, b1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = fast_exp2(mr[0][0] - b0), al1 = fast_exp2(mr[0][1] - b1);
      const float pc0 = fast_exp2(s0c - b0), pc1 = fast_exp2(s1c - b1);
      // l is summed over the 8 lanes of a column when the state is stored: add p once
      lr[0][0] = lr[0][0] * al0 + (n == 0 ? pc0 : 0.f);
      lr[0][1] = lr[0][1] * al1 + (n == 0 ? pc1 : 0.f);
      mr[0][0] = mn0;
      mr[0][1] = mn1;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int da = 32 * (mt >> 1) + 4 * n + 2 * (mt & 1);
        const float va = bf16_bits_to_float(nv[da]), vb = bf16_bits_to_float(nv[da + 1]);
        o[0][mt][0] = fmaf(pc0, va, o[0][mt][0] * al0);
        o[0][mt][1] = fmaf(pc1, va, o[0][mt][1] * al1);
        o[0][mt][2] = fmaf(pc0, vb, o[0][mt][2] * al0);
        o[0][mt][3] = fmaf(pc1, vb, o[0][mt][3] * al1);
      }
    } else if (warp == 1 && p.append) {
      const int page = __ldg(p.block_table + (size_t)w.b * p.max_pages + cur / p.page_size);
      if (page >= 0 && page < p.num_pages) {
        const int slot = cur % p.page_size;
        for (int plane = 0; plane < 2; ++plane) {
          // a token in slot 0 starts its page, which takes the step's formats
          const ol_plane_format pf = slot == 0 ? (plane == 0 ? p.new_fmt.k : p.new_fmt.v)
                                               : (plane == 0 ? fmts[page].k : fmts[page].v);
          const uint16_t* x = plane == 0 ? nk : nv;
          hp_encode_row_warp([&](int d) { return bf16_bits_to_float(x[d]); }, 128, pf,
                             hp_row(reinterpret_cast<uint8_t*>(p.pool), p.kv_heads, p.page_size, 128, page, plane,
                                    w.g, slot, pf.format));
          if (slot == 0 && w.g == 0 && lane == 0) {
            if (plane == 0)
              p.page_fmt[page].k = pf;
            else
              p.page_fmt[page].v = pf;
          }
        }
      } else if (lane == 0) {
        set_status(p.status, OL_DEVICE_GUARD);
      }
    }
  }

  float* merged = reinterpret_cast<float*>(stages + kStage);  // warp 0's second stage
  // each column group (a chunked step: each slice) merged and finished on its own
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    if (g >= nsl) break;
    if (g > 0) __syncthreads();  // the previous group's merge is done with the states and scratch
    store_warp_state<true>(reinterpret_cast<float*>(my_stages), ms, warp, o[g], mr[g][0], mr[g][1], lr[g][0],
                           lr[g][1]);
    merge_and_finish<NWARPS>(
        p, w, NWARPS, [&](int st) { return reinterpret_cast<const float*>(stages + st * STAGES * kStage); }, merged,
        nullptr, ms, CHUNK ? zs0 + g : -1);
  }
}

// ------------------------------------------------------------------ host

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// The pool as rows of `width` bytes (16-bit elements for width 256), boxes of 16 rows.
bool encode_width(CUtensorMap* map, void* base, uint64_t pool_bytes, int width) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const bool wide = width == 256;
  cuuint64_t dims[2] = {wide ? 128u : (cuuint64_t)width, pool_bytes / width};
  cuuint64_t strides[1] = {(cuuint64_t)width};
  cuuint32_t box[2] = {wide ? 64u : (cuuint32_t)width, kTok};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = width >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : width == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
  return fn(map, wide ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// decode steps: 6 warps x 2 stages, two CTAs per SM; chunked steps (two
// column groups, up to 255 registers): one CTA of kWarpsC warps per SM
constexpr int kWarps = 6, kStages = 2, kWarpsC = 8, kStagesC = 2;

template <bool CHUNK, bool DUP = false>
cudaError_t ensure_attrs() {
  constexpr int W = CHUNK ? kWarpsC : kWarps, S = CHUNK ? kStagesC : kStages;
  static cudaError_t state = cudaFuncSetAttribute(fast_hpaged_kernel<W, S, CHUNK, DUP>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  HpLayout<W, S, CHUNK ? 2 : 1>::kTotal);
  return state;
}

}  // namespace

bool fast_hpaged_supported(const AttnParams& p) {
  if (p.layout != OL_LAYOUT_HPAGED || p.head_dim != 128 || p.group > 8) return false;
  // a chunked step: query tokens share a CTA as extra columns (at most 8)
  if (p.nq > 1 && (p.tq < 1 || p.group * p.tq > 8)) return false;
  if (p.page_size % kTok != 0) return false;
  // TMA row coordinates are 32-bit: the 32-byte-row view has the most rows
  const unsigned long long rows32 = (unsigned long long)p.num_pages * p.kv_heads * p.page_size * 128 * 8 / 32;
  return rows32 < (1ull << 31);
}

int fast_hpaged_ctas_per_sm(bool chunk) {
  return chunk ? HpLayout<kWarpsC, kStagesC, 2>::kPerSm : HpLayout<kWarps, kStages>::kPerSm;
}

cudaError_t launch_fast_hpaged(const AttnParams& p, cudaStream_t s) {
  if (p.total_ctas <= 0) return cudaSuccess;
  const uint64_t bytes = (uint64_t)p.num_pages * p.kv_heads * p.page_size * 128 * 8;
  CUtensorMap maps[4];
  if (!encode_width(&maps[0], p.pool, bytes, 256) || !encode_width(&maps[1], p.pool, bytes, 128) ||
      !encode_width(&maps[2], p.pool, bytes, 64) || !encode_width(&maps[3], p.pool, bytes, 32))
    return cudaErrorInvalidValue;
  const bool chunk = p.nq > 1, dup = !chunk && p.group <= 4;
  cudaError_t e = chunk ? ensure_attrs<true>() : dup ? ensure_attrs<false, true>() : ensure_attrs<false>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  // a chunked step: pairs of slices of query tokens along x (a CTA carries two
  // slices' columns), the split plan's CTAs along y
  const int slices = (p.nq + p.tq - 1) / p.tq;
  cfg.gridDim = chunk ? dim3((slices + 1) / 2, p.total_ctas, 1) : dim3(p.total_ctas, 1, 1);
  cfg.blockDim = dim3((chunk ? kWarpsC : kWarps) * 32, 1, 1);
  cfg.dynamicSmemBytes = chunk ? HpLayout<kWarpsC, kStagesC, 2>::kTotal : HpLayout<kWarps, kStages>::kTotal;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (chunk)
    return cudaLaunchKernelEx(&cfg, fast_hpaged_kernel<kWarpsC, kStagesC, true>, maps[0], maps[1], maps[2], maps[3],
                              p);
  if (dup)  // the lo half of P^T in the free MMA columns
    return cudaLaunchKernelEx(&cfg, fast_hpaged_kernel<kWarps, kStages, false, true>, maps[0], maps[1], maps[2],
                              maps[3], p);
  return cudaLaunchKernelEx(&cfg, fast_hpaged_kernel<kWarps, kStages, false>, maps[0], maps[1], maps[2], maps[3], p);
}

}  // namespace ol
