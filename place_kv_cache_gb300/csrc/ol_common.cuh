// ol_common.cuh -- device helpers shared by the decode-step kernels:
// inline-PTX wrappers (mbarrier, bulk/tensor copies, ldmatrix, mma.sync,
// movmatrix, programmatic dependent launch), bf16/fp16 bit helpers, the
// CTA -> (row, kv head, split) mapping and the split-K merge.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ol_internal.h"
#include "ol_launch.h"

namespace ol {

constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at 2 GHz: bounded spin on mbarriers

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
// 1024-byte aligned start of a dynamic shared-memory buffer, kept as a
// shared-memory pointer (pointer arithmetic on the __shared__ array).
__device__ __forceinline__ uint8_t* align1024(uint8_t* smem_raw) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
  return smem_raw + ((1024u - (a & 1023u)) & 1023u);
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: returns false (and the caller records a device status) if the
// phase did not complete within kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
  return true;
}

// 2D tiled tensor copy global -> shared, completion on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
// 3D tiled tensor copy global -> shared, completion on an mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// The same with fp16 inputs.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------ bit helpers

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}
__device__ __forceinline__ float fp16_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ void set_status(int32_t* status, int32_t v) {
  if (status) atomicOr(reinterpret_cast<int*>(status), v);
}

// --------------------------------------------------------- CTA -> work map

// The work of one CTA: kv head g of row b, split s of nsplit; the tokens of
// the split's 16-token tiles (see row_split) clipped to the visible range
// [lo, hi); t_begin is a multiple of 16. A split may be empty when a short
// row's split count was rounded up to a whole cluster.
struct Work {
  int b, g, s, nsplit;
  int lo, hi;            // visible range of the row
  int t_begin, t_end;    // token range of this split (t_begin a multiple of 16)
  int first_cta;         // partial slot of split 0 of (b, g)
  int slot;              // this split's partial slot
  int next;              // stream-K: global tile of the CTA's next segment, -1 = none
  int valid;
};

// Computed by one full warp; every lane returns the same Work. CTAs go to the
// rows in the order `order` (a permutation of 0 .. batch - 1; NULL = row
// index order), the splits of one (row, kv head) on consecutive CTAs.
__device__ __forceinline__ Work map_cta_warp(const int32_t* __restrict__ lens, int batch, int kv_heads,
                                             int capacity, int window, int chunk, int cta,
                                             int32_t* status, int cluster = 1,
                                             const int16_t* __restrict__ order = nullptr) {
  const int lane = threadIdx.x & 31;
  Work w;
  w.valid = 0;
  w.b = w.g = w.s = 0;
  w.nsplit = 1;
  w.lo = w.hi = w.t_begin = w.t_end = 0;
  w.first_cta = w.slot = 0;
  w.next = -1;
  int running = 0;
  for (int base = 0; base < batch; base += 32) {
    const int i = base + lane;  // position in the launch order
    int b = i;
    if (order && i < batch) {
      b = order[i];
      if (b < 0 || b >= batch) {
        set_status(status, OL_DEVICE_GUARD);
        b = 0;
      }
    }
    int n = 0;
    if (i < batch) {
      n = lens[b];
      if (n < 0 || n > capacity) {
        set_status(status, OL_DEVICE_GUARD);
        n = n < 0 ? 0 : capacity;
      }
    }
    RowSplit rs = row_split(n, window, chunk, cluster);
    int cnt = (i < batch) ? rs.nsplit * kv_heads : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int total = __shfl_sync(0xffffffffu, incl, 31);
    if (cta < running + total) {
      int excl = incl - cnt;
      unsigned hit = __ballot_sync(0xffffffffu, cnt > 0 && cta >= running + excl && cta < running + incl);
      int src = __ffs(hit) - 1;
      int within = cta - running - __shfl_sync(0xffffffffu, excl, src);
      w.b = __shfl_sync(0xffffffffu, b, src);
      w.nsplit = __shfl_sync(0xffffffffu, rs.nsplit, src);
      w.lo = __shfl_sync(0xffffffffu, rs.lo, src);
      w.hi = __shfl_sync(0xffffffffu, rs.hi, src);
      int start = __shfl_sync(0xffffffffu, rs.start, src);
      int ntiles = __shfl_sync(0xffffffffu, rs.ntiles, src);
      w.g = within / w.nsplit;
      w.s = within % w.nsplit;
      w.t_begin = min(start + 16 * split_tile(w.s, ntiles, w.nsplit), w.hi);
      w.t_end = min(start + 16 * split_tile(w.s + 1, ntiles, w.nsplit), w.hi);
      w.first_cta = cta - w.s;
      w.slot = cta;
      w.valid = 1;
      return w;
    }
    running += total;
  }
  set_status(status, OL_DEVICE_GUARD);  // grid larger than the device-side plan
  return w;
}

// Grid roles. A decode step: x = CTA of the plan (clusters along x), y = the
// CUDA-core kernel's query-head block. A chunked step (nq > 1): x = query
// token, y = CTA of the plan (clusters along y), z = query-head block: the
// query tokens of one split are adjacent in launch order, so they run side by
// side and share the split's K/V tiles through L2.
__device__ __forceinline__ int cta_index(const AttnParams& p) { return p.nq > 1 ? blockIdx.y : blockIdx.x; }
__device__ __forceinline__ int query_index(const AttnParams& p) { return p.nq > 1 ? blockIdx.x : 0; }
__device__ __forceinline__ int head_block(const AttnParams& p) { return p.nq > 1 ? blockIdx.z : blockIdx.y; }

// A CTA's state columns: column c is query token c / group of the CTA's slice
// (tq tokens from slice_first) and head c % group; group * tq columns.
__device__ __forceinline__ int slice_tq(const AttnParams& p) { return p.nq > 1 && p.tq > 1 ? p.tq : 1; }
__device__ __forceinline__ int state_cols(const AttnParams& p) { return p.group * slice_tq(p); }
// slice zs (by default the launch's own, query_index)
__device__ __forceinline__ int slice_first(const AttnParams& p, int zs) { return zs * slice_tq(p); }
__device__ __forceinline__ int slice_first(const AttnParams& p) { return slice_first(p, query_index(p)); }
__device__ __forceinline__ int slice_tokens(const AttnParams& p, int zs) {
  return p.nq > 1 ? min(slice_tq(p), p.nq - slice_first(p, zs)) : 1;
}
__device__ __forceinline__ int slice_tokens(const AttnParams& p) { return slice_tokens(p, query_index(p)); }

// Chunked steps: query token z of every row sits at position hi - nq + z; its
// visible range ends there (causal inside the chunk) and starts window_q
// tokens before it. A CTA serves the slice's tokens: its range is clipped to
// the union of theirs (the first token's start to the last token's end), and
// the kernel masks each column to its own token's range. The plan's split
// stays.
// (A CTA serving slices za..zb takes the union of their ranges.)
__device__ __forceinline__ void slice_query(Work& w, const AttnParams& p, int za, int zb) {
  if (p.nq <= 1 || !w.valid) return;
  const int hi_first = w.hi - (p.nq - 1 - slice_first(p, za));
  const int hi_last = w.hi - (p.nq - 1 - (slice_first(p, zb) + slice_tokens(p, zb) - 1));
  const int lo = p.window_q < 0 ? w.lo : max(hi_first - 1 - p.window_q, 0);
  w.hi = hi_last;
  w.lo = max(w.lo, lo);
  w.t_end = min(w.t_end, hi_last);
  if (w.t_end < w.t_begin) w.t_end = w.t_begin;
}
__device__ __forceinline__ void slice_query(Work& w, const AttnParams& p) {
  slice_query(w, p, query_index(p), query_index(p));
}

// Length of row b as the kernels read it: clamped to [0, capacity], with a
// device status when it was out of range.
__device__ __forceinline__ int read_len(const int32_t* __restrict__ lens, int b, int capacity, int32_t* status) {
  int n = lens[b];
  if (n < 0 || n > capacity) {
    set_status(status, OL_DEVICE_GUARD);
    n = n < 0 ? 0 : capacity;
  }
  return n;
}

// Stream-K work. The 16-token tiles of all (row, kv head) units, in unit
// order u = b * kv_heads + g, are cut into `nctas` contiguous ranges of equal
// size; CTA c takes tiles [c*T/nctas, (c+1)*T/nctas) of the T tiles. Where its
// range crosses units it works in segments, one per unit. This returns the
// segment that starts at global tile x (x < 0: the CTA's first), with
//   slot = c + u (increasing along the tile order, so the segments of one
//   unit hold consecutive slots), first_cta = the slot of the unit's first
//   segment, nsplit = the unit's segment count, next = the start of the CTA's
//   following segment (-1: none).
// Computed by one full warp; every lane returns the same Work.
__device__ __forceinline__ Work map_streamk_warp(const int32_t* __restrict__ lens, int batch, int kv_heads,
                                                 int capacity, int window, int nctas, int cta, int x,
                                                 int32_t* status) {
  const int lane = threadIdx.x & 31;
  Work w;
  w.valid = 0;
  w.b = w.g = w.s = 0;
  w.nsplit = 1;
  w.lo = w.hi = w.t_begin = w.t_end = 0;
  w.first_cta = w.slot = 0;
  w.next = -1;
  long long T = 0;
  for (int base = 0; base < batch; base += 32) {
    const int b = base + lane;
    int nt = b < batch ? row_split(read_len(lens, b, capacity, status), window, 16).ntiles : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nt += __shfl_xor_sync(0xffffffffu, nt, o);
    T += nt;
  }
  T *= kv_heads;
  const long long g0 = (long long)cta * T / nctas, g1 = (long long)(cta + 1) * T / nctas;
  const long long xx = x < 0 ? g0 : x;
  if (xx >= g1) return w;  // an empty range, or past the CTA's last segment
  long long running = 0;  // first global tile of the chunk's first row
  for (int base = 0; base < batch; base += 32) {
    const int b = base + lane;
    RowSplit rs;
    rs.lo = rs.hi = rs.start = rs.ntiles = rs.nsplit = 0;
    if (b < batch) rs = row_split(read_len(lens, b, capacity, nullptr), window, 16);
    const long long cnt = b < batch ? (long long)rs.ntiles * kv_heads : 0;
    long long incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const long long total = __shfl_sync(0xffffffffu, incl, 31);
    if (xx < running + total) {
      const long long excl = incl - cnt;
      const unsigned hit = __ballot_sync(0xffffffffu, cnt > 0 && xx >= running + excl && xx < running + incl);
      const int src = __ffs(hit) - 1;
      const int nt = __shfl_sync(0xffffffffu, rs.ntiles, src);
      const int start = __shfl_sync(0xffffffffu, rs.start, src);
      const long long rb = running + __shfl_sync(0xffffffffu, excl, src);  // first tile of row b
      w.b = base + src;
      w.lo = __shfl_sync(0xffffffffu, rs.lo, src);
      w.hi = __shfl_sync(0xffffffffu, rs.hi, src);
      w.g = (int)((xx - rb) / nt);
      const long long au = rb + (long long)w.g * nt, bu = au + nt;  // the unit's tiles
      const long long se = bu < g1 ? bu : g1;
      w.t_begin = min(start + 16 * (int)(xx - au), w.hi);
      w.t_end = min(start + 16 * (int)(se - au), w.hi);
      const int cf = (int)(((au + 1) * nctas - 1) / T);  // CTA holding the unit's first tile
      const int cl = (int)((bu * nctas - 1) / T);        // and its last
      const int u = w.b * kv_heads + w.g;
      w.s = cta - cf;
      w.nsplit = cl - cf + 1;
      w.slot = cta + u;
      w.first_cta = cf + u;
      w.next = se < g1 ? (int)se : -1;
      w.valid = 1;
      return w;
    }
    running += total;
  }
  set_status(status, OL_DEVICE_GUARD);
  return w;
}

// -------------------------------------------------------- output + merge

__device__ __forceinline__ void store_out(void* out, int out_dtype, size_t idx, float v) {
  if (out_dtype == OL_F32)
    reinterpret_cast<float*>(out)[idx] = v;
  else
    reinterpret_cast<uint16_t*>(out)[idx] = float_to_bf16_bits(v);
}

// Split-K completion. A CTA holds, in shared memory, its merged state for the
// query heads [h0, h1) of its group and the dimensions [d0, d1):
// m[jl] (log2 domain), l[jl], o[jl * o_stride + (d - d0)] with jl = j - h0.
// Its result goes to partial slot `slot` of the `nslots` slots of (row, kv
// head), which start at `first_slot`. With one slot the CTA writes
// y = o / l directly; otherwise it stores the partial, takes a ticket, and the
// last of the `arrivals` CTAs of (row, kv head) merges all slots:
//   M = max_s m_s, L = sum_s l_s 2^(m_s - M), y = sum_s o_s 2^(m_s - M) / L.
// The merge first reduces (M, L) per head (one warp per head, lanes over the
// slots), then each output element reads its slots with independent loads.
// `scratch` is shared memory for 2 * state_cols(p) floats. The state's
// columns are (query token, head) pairs (see state_cols).
// Block-wide: every thread of the CTA must call it.
__device__ __forceinline__ void finish_split(const AttnParams& p, const Work& w, const float* sm_m,
                                             const float* sm_l, const float* sm_o, int o_stride, int h0,
                                             int h1, int d0, int d1, int slot, int first_slot, int nslots,
                                             int arrivals, int* sm_flag, float* scratch, int zs = -1) {
  const int D = p.head_dim;
  const int G = p.group;
  const int NC = state_cols(p);  // state columns: (query token, head) pairs
  const int tid = threadIdx.x;
  const int nthreads = blockDim.x;
  const int nh = h1 - h0, nd = d1 - d0;
  // a chunked step's slice zs: its own counters and partial slots; column c
  // goes to query token z0 + c / G, head c % G of y [B, Hq, nq, D]
  if (zs < 0) zs = query_index(p);  // the slice whose columns these are
  const int nq = p.nq > 1 ? p.nq : 1, z0 = slice_first(p, zs);
  const size_t head_base = (size_t)w.b * p.q_heads + (size_t)w.g * G;
  auto out_at = [&](int c, int d) -> size_t {
    if (nq == 1) return (head_base + c) * D + d;  // a decode step: column = head
    return ((head_base + c % G) * nq + z0 + c / G) * D + d;
  };
  const int c_live = G * slice_tokens(p, zs);  // columns past it belong to tokens beyond the chunk
  float* const partials =
      p.partials + (size_t)zs * ((size_t)p.batch * p.kv_heads + kMaxExtraSplits) * NC * (D + 2);  // max_ctas slots
  uint32_t* const counters = p.counters + (size_t)zs * p.batch * p.kv_heads;
  if (nslots == 1) {
    for (int i = tid; i < nh * nd; i += nthreads) {
      const int jl = i / nd, d = d0 + i % nd;
      const float l = sm_l[jl];
      const float y = l > 0.f ? sm_o[jl * o_stride + (d - d0)] / l : 0.f;
      if (h0 + jl < c_live) store_out(p.out, p.out_dtype, out_at(h0 + jl, d), y);
    }
    return;
  }
  float* sl = partials + (size_t)slot * NC * (D + 2);
  for (int i = tid; i < nh * (nd + 2); i += nthreads) {
    const int jl = i / (nd + 2), e = i % (nd + 2);
    if (e < 2) {
      if (d0 == 0) sl[(size_t)(h0 + jl) * (D + 2) + e] = e == 0 ? sm_m[jl] : sm_l[jl];
    } else {
      sl[(size_t)(h0 + jl) * (D + 2) + 2 + d0 + (e - 2)] = sm_o[jl * o_stride + (e - 2)];
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    unsigned* ctr = counters + (size_t)w.b * p.kv_heads + w.g;
    const unsigned prev = atomicAdd(ctr, 1u);
    const int last = (prev == (unsigned)(arrivals - 1));
    if (last) atomicExch(ctr, 0u);  // leave the ticket at zero for the next call
    *sm_flag = last;
  }
  __syncthreads();
  if (!*sm_flag) return;
  __threadfence();
  const float* base = partials + (size_t)first_slot * NC * (D + 2);
  const size_t stride = (size_t)NC * (D + 2);
  const int warp = tid >> 5, lane = tid & 31, nwarps = nthreads >> 5;
  for (int j = warp; j < NC; j += nwarps) {
    float M = -INFINITY;
    for (int s = lane; s < nslots; s += 32) M = fmaxf(M, __ldcg(base + s * stride + (size_t)j * (D + 2)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    if (M != -INFINITY)
      for (int s = lane; s < nslots; s += 32) {
        const float* ps = base + s * stride + (size_t)j * (D + 2);
        const float ms = __ldcg(ps);
        L += ms == -INFINITY ? 0.f : __ldcg(ps + 1) * fast_exp2(ms - M);
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) {
      scratch[2 * j] = M;
      scratch[2 * j + 1] = L;
    }
  }
  __syncthreads();
  for (int i = tid; i < c_live * D; i += nthreads) {
    const int j = i / D, d = i % D;
    const float M = scratch[2 * j], L = scratch[2 * j + 1];
    float acc = 0.f;
    if (M != -INFINITY) {
      const float* pj = base + (size_t)j * (D + 2);
#pragma unroll 8
      for (int s = 0; s < nslots; ++s) {
        const float ms = __ldcg(pj + s * stride);
        const float ov = __ldcg(pj + s * stride + 2 + d);
        acc += ms == -INFINITY ? 0.f : ov * fast_exp2(ms - M);
      }
    }
    store_out(p.out, p.out_dtype, out_at(j, d), L > 0.f ? acc / L : 0.f);
  }
}

// ------------------------------------------------------- thread-block clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}

// ----------------------------------------------------- INT4 quantization

// Quantize one token's D bf16 values (D a multiple of 32) into one INT4 row:
// per block of 32, fp16 scale and uint4 zero point (dynamic min-max or fixed
// parameters), code = sat[0,15](round_half_even(x / scale) + zp) in IEEE fp32.
// Executed by one full warp; lane i handles element i of each block.
__device__ __forceinline__ void int4_quantize_row_warp(const uint16_t* __restrict__ x, int D, int mode,
                                                       float fixed_scale, int fixed_zp,
                                                       uint8_t* __restrict__ codes_row,
                                                       uint16_t* __restrict__ scales_row,
                                                       uint8_t* __restrict__ zps_row) {
  const int lane = threadIdx.x & 31;
  const int nb = D / 32;
  uint32_t zp_acc = 0;  // lane 0 collects the packed zero points
  for (int blk = 0; blk < nb; ++blk) {
    float v = bf16_bits_to_float(x[blk * 32 + lane]);
    float s;
    int zp;
    uint16_t sbits;
    if (mode == OL_Q_FIXED) {
      sbits = __half_as_ushort(__float2half_rn(fixed_scale));
      s = fp16_bits_to_float(sbits);
      zp = fixed_zp;
    } else {
      float lo = fminf(v, 0.f), hi = fmaxf(v, 0.f);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
      }
      float s32 = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
      sbits = __half_as_ushort(__float2half_rn(s32));
      s = fp16_bits_to_float(sbits);
      if (s == 0.f) {
        sbits = __half_as_ushort(__float2half_rn(1.0f));
        s = 1.0f;
      }
      float z = rintf(__fdiv_rn(-lo, s));
      z = fminf(fmaxf(z, 0.f), 15.f);
      zp = static_cast<int>(z);
    }
    float r = __fadd_rn(rintf(__fdiv_rn(v, s)), static_cast<float>(zp));
    r = fminf(fmaxf(r, 0.f), 15.f);
    uint32_t code = static_cast<uint32_t>(r);
    uint32_t hi_code = __shfl_down_sync(0xffffffffu, code, 1);
    if ((lane & 1) == 0) codes_row[blk * 16 + lane / 2] = static_cast<uint8_t>(code | (hi_code << 4));
    if (lane == 0) {
      scales_row[blk] = sbits;
      zp_acc |= static_cast<uint32_t>(zp) << (4 * (blk & 1));
      if ((blk & 1) == 1 || blk == nb - 1) {
        zps_row[blk / 2] = static_cast<uint8_t>(zp_acc);
        zp_acc = 0;
      }
    }
  }
}

}  // namespace ol
