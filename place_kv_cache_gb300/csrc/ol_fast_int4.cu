// ol_fast_int4.cu -- tensor-core decode attention (and fused quantize-append)
// over the INT4 blockwise-affine cache with head_dim 128 and a GQA group of at
// most 8: codes [2, B, Hkv, C, 64] (two uint4 per byte, low nibble first),
// fp16 scales [2, B, Hkv, C, 4] and zero points [2, B, Hkv, C, 2] (two uint4
// per byte), one (scale, zero point) per block of 32 dims.
//
// Same decomposition as the bf16 kernel (one CTA per (row, kv head, split),
// warps over 16-token tiles, shared merge). A ring of stages holds NWARPS
// consecutive tiles each, one per warp; a stage arrives by three 3-D tensor
// copies that each cover the K and the V plane: codes (SWIZZLE_64B, 64-byte
// rows: conflict-free reads), scales and zero points. The last warp to finish
// with a stage issues its refill.
// Dequantization happens in registers and is exact:
//   S^T: one fp32 accumulator per 32-dim block b. The codes are fp16
//        operands as they lie in memory (a masked nibble is the subnormal
//        c * 2^-24, or 16c * 2^-24 one nibble up, which q absorbs as q / 16);
//        one more k-step adds zp_K * (-sum of the block's q). Then
//        s = sum_b scale_K[t,b] * acc_b.
//   O^T: the V code words masked in place as fp16 subnormals (as for K)
//        minus the zero point (an exact subnormal difference), the V scale
//        folded into P^T per block, P^T as fp16 hi + lo under a warp-uniform
//        power of two.
// The token being appended (fused step) takes part uncompressed from new_kv as
// one extra merge state, and is quantized into the cache by the same CTA.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "ol_merge.cuh"

namespace ol {
namespace {

constexpr int kTok = 16;
constexpr uint32_t kLoNib = 0x000F000Fu;  // nibble in bits 0..3 of both 16-bit halves
constexpr uint32_t kHiNib = 0x00F000F0u;  // nibble in bits 4..7 of both halves
constexpr int kStateBytes = 8 * kOStride * 4;  // one warp's [8][kOStride] fp32 state
constexpr float kLazy = 8.f;  // log2 headroom of the lazy softmax maximum
constexpr int kNoExp = -1000;  // no V exponent chosen yet (no tile seen)

// A stage: NWARPS tiles of 16 tokens. Byte offsets (NW = NWARPS):
//   K codes [16NW][64] @0, V codes @1024NW, K scales [16NW][4] fp16 @2048NW,
//   V scales @2176NW, K zero points [16NW][2] @2304NW, V zero points @2336NW.
template <int NW>
struct Int4Stage {
  static constexpr int kCodes = 1024 * NW;  // one plane's codes
  static constexpr int kOffSk = 2048 * NW, kOffSv = 2176 * NW, kOffZk = 2304 * NW, kOffZv = 2336 * NW;
  static constexpr int kTx = 2368 * NW;                   // bytes the three copies deliver
  static constexpr int kBytes = (kTx + 1023) / 1024 * 1024;  // 1024-aligned stride
};

template <int NWARPS, int STAGES, int NG = 1>
struct Int4Layout {
  static constexpr int kStages = STAGES * Int4Stage<NWARPS>::kBytes;
  // extra state O of each column group, then one region that is either the
  // CTA-merged state (no cluster) or the cluster receive buffers + cmerged
  // (cluster): never both
  static constexpr int kUnion = (1024 + 2 * 128 + 8 * 64) * 4 > kStateBytes ? (1024 + 2 * 128 + 8 * 64) * 4
                                                                         : kStateBytes;
  static constexpr int kExtra = NG * kStateBytes + kUnion;
  static constexpr int kBars = STAGES * 8 + STAGES * 4;  // full barriers, release counters
  static constexpr int kMisc = 256 + (NWARPS + NG) * 8 * 4 * 2 + 8 * 4 * 6 + 16 * 4 + 2 * 16 * 8 * 4 + 16;
  static constexpr int kTotal = 1024 + kStages + kExtra + (kBars + 15) / 16 * 16 + kMisc;
  // CTAs per SM: shared memory, and registers (one column group: up to 16
  // warps per SM, i.e. 128 registers per thread at 8 warps per CTA and up to
  // 168 at 6; two groups take up to 255, one CTA per SM)
  static constexpr int kBySmem = (228 * 1024) / (kTotal + 1024) > 0 ? (228 * 1024) / (kTotal + 1024) : 1;
  static constexpr int kByRegs = NG > 1 ? 8 / NWARPS : 16 / NWARPS;
  static constexpr int kPerSm = kBySmem < kByRegs ? kBySmem : (kByRegs > 0 ? kByRegs : 1);
  static_assert(kStages >= NWARPS * kStateBytes, "the warps' states fit in the stages");
};

// fp16 pair difference (exact for the subnormal code and zero-point values used here)
__device__ __forceinline__ uint32_t hsub2_f16(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t x) {
  return __half22float2(*reinterpret_cast<__half2*>(&x));
}
// packed pairs of fp32 (one instruction for two lanes' columns 2c, 2c + 1)
__device__ __forceinline__ float2 bc2(float x) { return make_float2(x, x); }
// byte offset of logical byte x of 64-byte row r in a SWIZZLE_64B tile
__device__ __forceinline__ int swz64(int r, int x) {
  return r * 64 + ((((x >> 4) ^ (r >> 1)) & 3) << 4) + (x & 15);
}

// CHUNK: a chunked step's attention (grid x = slice of query tokens, y = the
// plan's CTA): state columns are (query token, head) pairs, each masked to its
// token's window; the history ends where the chunk starts, and the chunk's
// tokens take part uncompressed from new_kv as one causal extra state per
// column. Its own instantiation: the decode kernel keeps its own code.
// DUP (a decode step with at most 4 heads per kv head): MMA columns 4..7
// repeat the heads of columns 0..3, so the two halves of P^T (fp16 hi and lo)
// travel in one MMA, hi in columns 0..3 and lo in 4..7, added when the state
// is stored; and the V zero point leaves the code operands: its term
// sum_t P'[t] * zp[t] is one fp32 sum per (block, column), subtracted at the end.
template <int NWARPS, int STAGES, bool CHUNK = false, bool DUP = false>
__global__ void __launch_bounds__(NWARPS * 32, Int4Layout<NWARPS, STAGES, CHUNK ? 2 : 1>::kPerSm)
    fast_int4_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_scales,
                     const __grid_constant__ CUtensorMap tm_zps, const __grid_constant__ AttnParams p) {
  static_assert(!(CHUNK && DUP), "duplicated columns serve a decode step only");
  constexpr int NG = CHUNK ? 2 : 1;  // column groups a warp carries (a chunked step: two slices)
  using L = Int4Layout<NWARPS, STAGES, NG>;
  using S = Int4Stage<NWARPS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* stages = smem;
  float* extra_o = reinterpret_cast<float*>(smem + L::kStages);  // [NG][8][kOStride]
  float* merged = extra_o + NG * 8 * kOStride;  // no cluster: the CTA state
  float* recv = merged;                    // cluster: receive buffers, then cmerged
  float* cmerged = recv + 1024 + 256;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kStages + L::kExtra);
  int* freed = reinterpret_cast<int*>(smem + L::kStages + L::kExtra + STAGES * 8);  // warps done per stage
  Work* sw = reinterpret_cast<Work*>(smem + L::kStages + L::kExtra + (L::kBars + 15) / 16 * 16);
  float* misc = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(sw) + 256);
  MergeScratch ms;
  ms.wm = misc;                        // [NWARPS + NG][8]: warps, then the extra states
  ms.wl = ms.wm + (NWARPS + NG) * 8;   // [NWARPS + NG][8]
  ms.m = ms.wl + (NWARPS + NG) * 8;
  ms.l = ms.m + 8;
  ms.cm = ms.l + 8;
  ms.cl = ms.cm + 8;
  ms.scr = ms.cl + 8;
  ms.cw = ms.scr + 16;
  ms.wt = ms.cw + 16 * 8;
  ms.flag = reinterpret_cast<int*>(ms.wt + 16 * 8);
  ms.recv_o = recv;
  ms.recv_m = recv + 1024;
  ms.recv_l = recv + 1024 + 128;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int CS = p.cluster;
  const uint32_t bar0 = smem_u32(bars);
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tm_codes);
    prefetch_tensormap(&tm_scales);
    prefetch_tensormap(&tm_zps);
    for (int st = 0; st < STAGES; ++st) {
      mbar_init(bar0 + 8 * st, 1);
      freed[st] = 0;
    }
    fence_mbar_init();
  }
  if (!p.inline_lens) pdl_wait();
  const int32_t* lens = p.inline_lens ? p.lens_inline : p.lens;
  int32_t* const lens_status = p.inline_lens ? nullptr : p.status;
  // a chunked step's CTA serves NG consecutive slices of query tokens, zs0 .. zs0 + nsl - 1
  const int nslices = CHUNK ? (p.nq + slice_tq(p) - 1) / slice_tq(p) : 1;
  const int zs0 = CHUNK ? NG * query_index(p) : 0;
  const int nsl = CHUNK ? min(NG, nslices - zs0) : 1;
  int jbase = 0;  // stages consumed by earlier segments: ring slot and mbarrier phase
  int next = -1;  // stream-K: global tile where the next segment starts
  // One pass per segment: a split of one (row, kv head). Without stream-K a
  // CTA has one segment.
  for (int seg = 0;; ++seg) {
  if (seg > 0) __syncthreads();  // the previous segment's Work and states are done with
  if (warp == 0) {
    Work w = p.streamk ? map_streamk_warp(lens, p.batch, p.kv_heads, p.capacity, p.window, p.total_ctas,
                                          cta_index(p), next, lens_status)
                       : map_cta_warp(lens, p.batch, p.kv_heads, p.capacity, p.window, p.chunk, cta_index(p),
                                      lens_status, CS, p.inline_lens && p.ordered ? p.row_order : nullptr);
    if (CHUNK) slice_query(w, p, zs0, zs0 + nsl - 1);
    if (lane == 0) *sw = w;
  }
  __syncthreads();
  const Work w = *sw;
  if (!w.valid && (seg > 0 || CS == 1)) {  // a cluster's idle CTAs still take part in its merge
    if (seg == 0 && p.inline_lens) pdl_wait();
    return;
  }

  const int G = p.group;
  const int C = p.capacity;
  const int nsub = w.valid ? (w.t_end - w.t_begin + kTok - 1) / kTok : 0;  // tiles of the CTA
  const int nstage = (nsub + NWARPS - 1) / NWARPS;                              // stages of the CTA
  // a decode step reads each byte once; a chunked step's slices (adjacent in
  // launch order) read the same tiles, the later ones from L2
  const uint64_t pol = CHUNK ? policy_evict_normal() : policy_evict_first();
  const int row0 = (w.b * p.kv_heads + w.g) * C;  // row of token 0 within a plane
  const int rowK0 = row0, rowV0 = p.batch * p.kv_heads * C + row0;

  // Stage j (tiles NWARPS*j ..) into ring slot j % STAGES: codes, scales and
  // zero points of tokens t .. t + 16*NWARPS - 1 of both planes. Boxes that run
  // past the CTA's range read tokens nobody uses (or the fill value past the
  // end of the arrays).
  auto issue = [&](int j) {
    const int st = (jbase + j) % STAGES;
    const uint32_t dst = smem_u32(stages + st * S::kBytes);
    const uint32_t bar = bar0 + 8 * st;
    const int r = row0 + w.t_begin + j * NWARPS * kTok;  // multiple of 16
    mbar_arrive_expect_tx(bar, S::kTx);
    tma_load_3d(dst, &tm_codes, 0, r, 0, bar, pol);
    tma_load_3d(dst + S::kOffSk, &tm_scales, 0, r >> 1, 0, bar, pol);
    tma_load_3d(dst + S::kOffZk, &tm_zps, 0, r >> 3, 0, bar, pol);
  };
  const int pre = nstage < STAGES ? nstage : STAGES;
  if (seg == 0) {
    if (p.early && threadIdx.x == 0)
      for (int j = 0; j < pre; ++j) issue(j);
    if (p.inline_lens) pdl_wait();
    pdl_launch_dependents();
    if (!p.early && threadIdx.x == 0)
      for (int j = 0; j < pre; ++j) issue(j);
  } else if (threadIdx.x == 0) {
    fence_proxy_async_smem();  // the previous segment's generic use of the stages first
    for (int j = 0; j < pre; ++j) issue(j);
  }

  // K side operands. The codes enter the tensor cores as fp16 subnormals: a
  // 16-bit lane holding c in bits 0..3 is c * 2^-24, in bits 4..7 it is
  // 16c * 2^-24, both exact, so one mask yields two operands. q is converted
  // to fp16 scaled by 2^eq, with eq chosen to put max |q| in [2^9, 2^10)
  // (exact: bf16 values are fp16 values times a power of two, unless tiny).
  // Lane (c, n) holds q[n][32b + 8c + i], i = 0..7, in the nibble order of a
  // code word:  k-step 0 of block b: b0 = (i0, i4), b1 = (i1, i5) / 16,
  //             k-step 1:            b0 = (i2, i6), b1 = (i3, i7) / 16.
  // A third k-step per block adds zp * (-Q_b), Q_b the sum of the block's
  // fp16 q carried as two fp16 (rows 0 and 1 of lane c = 0).
  // Column group g (a chunked step: slice zs0 + g) has its own q operands,
  // scores, softmax state and O; the code-word operands of a tile serve all.
  const int c = lane & 3, n = lane >> 2;
  const int ncol = DUP ? (n & 3) : n;  // the head (or token-head pair) of MMA column n
  uint32_t qf[NG][4][2][2], qz[NG][4];
  float sfac;  // converts an accumulator (units 2^-24 * 2^eq) to the exp2 domain
  // A chunked step's column n of group g is head n % G of slice zs0 + g's query token n / G.
  {
    float qv[NG][4][8];
    float mx = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const int zs = zs0 + g;
      const bool live = g < nsl && ncol < (CHUNK ? G * slice_tokens(p, zs) : G) && w.valid;
      const int nl = live ? ncol : 0;
      const uint16_t* qp = reinterpret_cast<const uint16_t*>(p.q) +
                           (CHUNK ? (((size_t)w.b * p.q_heads + (size_t)w.g * G + nl % G) * p.nq + slice_first(p, zs) +
                                     nl / G) * 128
                                  : ((size_t)w.b * p.q_heads + (size_t)w.g * G + nl) * 128);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint4 v = live ? __ldg(reinterpret_cast<const uint4*>(qp + 32 * b + 8 * c)) : make_uint4(0, 0, 0, 0);
        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          qv[g][b][2 * k] = __uint_as_float(wd[k] << 16);
          qv[g][b][2 * k + 1] = __uint_as_float(wd[k] & 0xffff0000u);
          mx = fmaxf(mx, fmaxf(fabsf(qv[g][b][2 * k]), fabsf(qv[g][b][2 * k + 1])));
        }
      }
    }
    mx = warp_max(mx);
    int eq = 0;
    if (mx > 0.f && mx <= 3.0e38f) {
      int e2;
      frexpf(mx, &e2);  // mx = f * 2^e2, f in [0.5, 1)
      eq = min(100, max(-100, 10 - e2));
    }
    const float qscale = ldexpf(1.f, eq);
    sfac = ldexpf(p.scale_log2, 24 - eq);
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float qh[8];
        float qs = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          qh[i] = __half2float(__float2half_rn(qv[g][b][i] * qscale));
          qs += qh[i];
        }
        qf[g][b][0][0] = pack_f16x2(qh[0], qh[4]);
        qf[g][b][0][1] = pack_f16x2(qh[1] * 0.0625f, qh[5] * 0.0625f);
        qf[g][b][1][0] = pack_f16x2(qh[2], qh[6]);
        qf[g][b][1][1] = pack_f16x2(qh[3] * 0.0625f, qh[7] * 0.0625f);
        qs += __shfl_xor_sync(0xffffffffu, qs, 1);
        qs += __shfl_xor_sync(0xffffffffu, qs, 2);
        const float qhi = __half2float(__float2half_rn(qs));
        // blocks 1 and 3 meet their zero point in bits 4..7 (16 zp): Q / 16
        const float zf = (b & 1) ? 0.0625f : 1.f;
        qz[g][b] = c == 0 ? pack_f16x2(-qhi * zf, -(qs - qhi) * zf) : 0u;
      }
  }
  // The code words come from ldmatrix: the 16 bytes of block b in a token's
  // 64-byte row are one 8 x b16 matrix row, b16 k holding dims 32b + 4k .. +3.
  // Matrix m of a x4 load covers tokens 8(m & 1) .. +7 of block 2h + (m >> 1)
  // (block pair h); lane l gives the address of row l % 8 of matrix l / 8 in
  // the warp's tile (rows 16*warp .. +15 of each plane, 64-byte swizzle).
  //   K, plain: lane (c, n) gets bytes 4c .. 4c+3 of token n (matrices 0, 2)
  //     and of token n + 8 (1, 3): the A words of S^T = K q^T.
  //   V, transposed: lane (c, n) gets the b16 n (dims 32b + 4n .. +3) of
  //     tokens 2c and 2c + 1 (matrices 0, 2; tokens 2c + 8, 2c + 9 from 1, 3)
  //     in the low and high halves: the A words of O^T += V^T P^T.
  uint32_t kaddr[2], vaddr[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int tok = (lane & 7) + 8 * ((lane >> 3) & 1), blk = 2 * h + (lane >> 4);
    kaddr[h] = 1024 * warp + swz64(tok, 16 * blk);
    vaddr[h] = S::kCodes + 1024 * warp + swz64(tok, 16 * blk);
  }

  float o[NG][8][4];
  float mr[NG][2], lr[NG][2];  // running maximum and sum of the lane's columns 2c, 2c + 1
#pragma unroll
  for (int g = 0; g < NG; ++g) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[g][mt][0] = o[g][mt][1] = o[g][mt][2] = o[g][mt][3] = 0.f;
    mr[g][0] = mr[g][1] = -INFINITY;
    lr[g][0] = lr[g][1] = 0.f;
  }
  int ev = kNoExp;  // O is held in units of 2^(ev - 24) (V side, see the tile)
  float pe = 0.f;   // 2^ev
  // the running maximum as the exp2 offset: 0 while no score is finite
  float rz[NG][2];
#pragma unroll
  for (int g = 0; g < NG; ++g) rz[g][0] = rz[g][1] = 0.f;
  // DUP: the V zero-point term of the lane's columns 2c, 2c + 1 per block b,
  // over its tokens n, n + 8, times 16^b (units of O times 2^24)
  float zc[DUP ? 4 : 1][2];
#pragma unroll
  for (int b = 0; b < (DUP ? 4 : 1); ++b) zc[b][0] = zc[b][1] = 0.f;
  // DUP: 1 on the lanes of columns 4..7, whose P^T operand is the lo half
  const float hsel = DUP && c >= 2 ? 1.f : 0.f;
  // tokens below codes_hi come from the codes: a decode step's history ends
  // before its current token, a chunked step's before its chunk (w.hi is one
  // past the last query token of the CTA's last slice, at codes_hi + zlast)
  const int zlast = CHUNK ? slice_first(p, zs0 + nsl - 1) + slice_tokens(p, zs0 + nsl - 1) - 1 : 0;
  const int codes_hi = CHUNK ? w.hi - 1 - zlast : (p.cur_from_new ? w.hi - 1 : w.hi);
  const int t_stop = min(w.t_end, codes_hi);
  // visible history of the lane's columns 2c, 2c + 1 of each group (chunked
  // step): from its query token's window start; a tile is FULL only if it
  // starts at or past every column's start (the last token has the latest one)
  int clo[NG][2], lo_full = w.lo;
#pragma unroll
  for (int g = 0; g < NG; ++g) clo[g][0] = clo[g][1] = w.lo;
  if (CHUNK && p.window_q >= 0) {
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const int zs = zs0 + min(g, nsl - 1);
      const int last = slice_tokens(p, zs) - 1;
      const int base = codes_hi + slice_first(p, zs);  // position of the slice's first query token
      clo[g][0] = max(w.lo, base + min((2 * c) / G, last) - p.window_q);
      clo[g][1] = max(w.lo, base + min((2 * c + 1) / G, last) - p.window_q);
    }
    lo_full = max(w.lo, codes_hi + zlast - p.window_q);
  }

  // One 16-token tile in stage base sg. FULL: every token of the tile is
  // visible (no masking of scores or scales).
  auto tile = [&](const uint32_t sg, const int t0, auto full_tag) {
    constexpr bool FULL = decltype(full_tag)::value;
    const uint32_t ksc = sg + S::kOffSk + 128 * warp, vsc = sg + S::kOffSv + 128 * warp;
    const uint32_t kz = sg + S::kOffZk + 32 * warp, vz = sg + S::kOffZv + 32 * warp;
    bool va = true, vb = true;  // the lane's S^T rows (tokens n, n + 8) are visible (to some column)
    if (!FULL) {
      va = t0 + n >= w.lo && t0 + n < t_stop;
      vb = t0 + n + 8 >= w.lo && t0 + n + 8 < t_stop;
    }

    // ---- S^T = K q^T, one accumulator per 32-dim block (and column group)
    const uint32_t zda = lds_u16(kz + 2 * n) * 0x10001u, zdb = lds_u16(kz + 2 * n + 16) * 0x10001u;
    uint32_t kw[4][2];  // [block][tokens n, n + 8]
    ldsm_x4(sg + kaddr[0], kw[0][0], kw[0][1], kw[1][0], kw[1][1]);
    ldsm_x4(sg + kaddr[1], kw[2][0], kw[2][1], kw[3][0], kw[3][1]);
    float sacc[NG][4][4];
    // zero points of blocks 0 / 1 in bits 0..3 / 4..7 of each half, blocks 2 / 3 one byte up
    const uint32_t zda8 = zda >> 8, zdb8 = zdb >> 8;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t wa = kw[b][0], wb = kw[b][1];
      const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
      const uint32_t a0 = wa & kLoNib, a1 = wb & kLoNib, a2 = wa & kHiNib, a3 = wb & kHiNib;
      const uint32_t c0 = wa8 & kLoNib, c1 = wb8 & kLoNib, c2 = wa8 & kHiNib, c3 = wb8 & kHiNib;
      const uint32_t zm = (b & 1) ? kHiNib : kLoNib;  // block b's nibble in place (x16 for odd b)
      const uint32_t za = (b < 2 ? zda : zda8) & zm, zb = (b < 2 ? zdb : zdb8) & zm;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        sacc[g][b][0] = sacc[g][b][1] = sacc[g][b][2] = sacc[g][b][3] = 0.f;
        mma_f16_16816(sacc[g][b], a0, a1, a2, a3, qf[g][b][0][0], qf[g][b][0][1]);
        mma_f16_16816(sacc[g][b], c0, c1, c2, c3, qf[g][b][1][0], qf[g][b][1][1]);
        mma_f16_16816(sacc[g][b], za, zb, za, zb, qz[g][b], 0u);
      }
    }
    const uint2 ska = lds_v2(ksc + 8 * n), skb = lds_v2(ksc + 8 * n + 64);
    const float2 ka01 = half2_bits_to_float2(ska.x), ka23 = half2_bits_to_float2(ska.y);
    const float2 kb01 = half2_bits_to_float2(skb.x), kb23 = half2_bits_to_float2(skb.y);
    float pw[NG][4];  // weights: (token n, column 2c), (n, 2c + 1), (n + 8, 2c), (n + 8, 2c + 1)
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const float(&sc)[4][4] = sacc[g];
      // columns (2c, 2c + 1) of tokens n and n + 8 as pairs
      float2 sa2 = __fmul2_rn(bc2(ka01.x), make_float2(sc[0][0], sc[0][1]));
      float2 sb2 = __fmul2_rn(bc2(kb01.x), make_float2(sc[0][2], sc[0][3]));
      sa2 = __ffma2_rn(bc2(ka01.y), make_float2(sc[1][0], sc[1][1]), sa2);
      sb2 = __ffma2_rn(bc2(kb01.y), make_float2(sc[1][2], sc[1][3]), sb2);
      sa2 = __ffma2_rn(bc2(ka23.x), make_float2(sc[2][0], sc[2][1]), sa2);
      sb2 = __ffma2_rn(bc2(kb23.x), make_float2(sc[2][2], sc[2][3]), sb2);
      sa2 = __ffma2_rn(bc2(ka23.y), make_float2(sc[3][0], sc[3][1]), sa2);
      sb2 = __ffma2_rn(bc2(kb23.y), make_float2(sc[3][2], sc[3][3]), sb2);
      sa2 = __fmul2_rn(sa2, bc2(sfac));
      sb2 = __fmul2_rn(sb2, bc2(sfac));
      float s00 = sa2.x, s01 = sa2.y, s10 = sb2.x, s11 = sb2.y;
      if (!FULL) {
        if (CHUNK) {  // each column from its own window start
          s00 = va && t0 + n >= clo[g][0] ? s00 : -INFINITY;
          s01 = va && t0 + n >= clo[g][1] ? s01 : -INFINITY;
          s10 = vb && t0 + n + 8 >= clo[g][0] ? s10 : -INFINITY;
          s11 = vb && t0 + n + 8 >= clo[g][1] ? s11 : -INFINITY;
        } else {
          s00 = va ? s00 : -INFINITY;
          s01 = va ? s01 : -INFINITY;
          s10 = vb ? s10 : -INFINITY;
          s11 = vb ? s11 : -INFINITY;
        }
      }

      // ---- online softmax (exp2 domain) with a lazy maximum: the weights are
      // taken against the running maximum m as long as no score exceeds it by
      // more than kLazy (weights stay below 2^kLazy); only then is the tile's
      // maximum reduced across the lanes and the state rescaled
      if (__any_sync(0xffffffffu, fmaxf(s00, s10) > mr[g][0] + kLazy || fmaxf(s01, s11) > mr[g][1] + kLazy)) {
        float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(mr[g][0], mx0), mn1 = fmaxf(mr[g][1], mx1);
        const float al0 = mn0 == mr[g][0] ? 1.f : fast_exp2(mr[g][0] - mn0);
        const float al1 = mn1 == mr[g][1] ? 1.f : fast_exp2(mr[g][1] - mn1);
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
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            zc[b][0] *= al0;
            zc[b][1] *= al1;
          }
        }
        mr[g][0] = mn0;
        mr[g][1] = mn1;
        rz[g][0] = mn0 == -INFINITY ? 0.f : mn0;
        rz[g][1] = mn1 == -INFINITY ? 0.f : mn1;
      }
      const float r0 = rz[g][0], r1 = rz[g][1];
      pw[g][0] = fast_exp2(s00 - r0);
      pw[g][1] = fast_exp2(s01 - r1);
      pw[g][2] = fast_exp2(s10 - r0);
      pw[g][3] = fast_exp2(s11 - r1);
      lr[g][0] += pw[g][0] + pw[g][2];
      lr[g][1] += pw[g][1] + pw[g][3];
    }

    // ---- O^T += V^T P^T, block by block. A = the V code words masked in
    // place: fp16 subnormals c * 2^-24 (rows n: dims 32b + 4n + 2h), or
    // 16c * 2^-24 for a code in bits 4..7 (rows n + 8: dims 32b + 4n + 2h + 1,
    // which therefore hold 16 O and are scaled back when the state is
    // stored), minus the zero point in the same units: (c - zp) * 2^-24, a
    // subnormal difference, exact. B = P^T times the token's V scale and
    // 2^ev as fp16 hi + lo (about 22 significant bits per weight: the error
    // does not grow with the size of the values). ev is warp-uniform:
    // 2^kLazy * (largest V scale of the tile) * 2^ev stays below 2^15, and O
    // is held in units of 2^(ev - 24); it is rescaled only when the tile
    // needs a smaller ev, or a much larger one.
    const uint2 sva = lds_v2(vsc + 8 * n), svb = lds_v2(vsc + 8 * n + 64);
    uint32_t sa0 = sva.x, sa1 = sva.y, sb0 = svb.x, sb1 = svb.y;
    if (!FULL) {  // a hidden token's scale may be anything: its weight is exactly 0
      if (!va) sa0 = sa1 = 0u;
      if (!vb) sb0 = sb1 = 0u;
    }
    {
      // largest scale of the tile (positive fp16 order as unsigned integers)
      uint32_t mx = __vmaxu2(__vmaxu2(sa0, sa1), __vmaxu2(sb0, sb1));
      mx = __reduce_max_sync(0xffffffffu, max(mx & 0xffffu, mx >> 16));
      const int e_want = 21 - (int)((mx >> 10) & 31u);  // scale < 2^(field - 14)
      if (e_want < ev || e_want > ev + 6) {
        if (ev != kNoExp) {
          const float f = ldexpf(1.f, e_want - ev);
#pragma unroll
          for (int g = 0; g < NG; ++g)
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              o[g][mt][0] *= f;
              o[g][mt][1] *= f;
              o[g][mt][2] *= f;
              o[g][mt][3] *= f;
            }
          if constexpr (DUP) {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              zc[b][0] *= f;
              zc[b][1] *= f;
            }
          }
        }
        ev = e_want;
        pe = __int_as_float((127 + e_want) << 23);  // e_want in [-10, 21]
      }
    }
    float pa[NG][4];
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int k = 0; k < 4; k += 2) {
        const float2 x = __fmul2_rn(make_float2(pw[g][k], pw[g][k + 1]), bc2(pe));
        pa[g][k] = x.x;
        pa[g][k + 1] = x.y;
      }
    const float2 va01 = half2_bits_to_float2(sa0), va23 = half2_bits_to_float2(sa1);
    const float2 vb01 = half2_bits_to_float2(sb0), vb23 = half2_bits_to_float2(sb1);
    uint32_t vw[4][2];  // [block][tokens (2c, 2c+1), (2c+8, 2c+9)]
    ldsm_x4_trans(sg + vaddr[0], vw[0][0], vw[0][1], vw[1][0], vw[1][1]);
    ldsm_x4_trans(sg + vaddr[1], vw[2][0], vw[2][1], vw[3][0], vw[3][1]);
    if constexpr (DUP) {
      // zero points of the lane's weights' tokens n and n + 8 (all four
      // blocks in one 16-bit word each)
      const uint32_t zn = lds_u16(vz + 2 * n), zn8 = lds_u16(vz + 2 * n + 16);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float sca = b == 0 ? va01.x : b == 1 ? va01.y : b == 2 ? va23.x : va23.y;
        const float scb = b == 0 ? vb01.x : b == 1 ? vb01.y : b == 2 ? vb23.x : vb23.y;
        // P^T times the V scale, columns (2c, 2c + 1) of tokens n and n + 8 as pairs
        const float2 qa = __fmul2_rn(make_float2(pa[0][0], pa[0][1]), bc2(sca));
        const float2 qb = __fmul2_rn(make_float2(pa[0][2], pa[0][3]), bc2(scb));
        // hi on the lanes of columns 0..3, lo = what hi leaves on those of 4..7
        const float2 f0 = half2_bits_to_float2(pack_f16x2(qa.x, qa.y));
        const float2 f1 = half2_bits_to_float2(pack_f16x2(qb.x, qb.y));
        const float2 y0 = __ffma2_rn(bc2(-hsel), f0, qa), y1 = __ffma2_rn(bc2(-hsel), f1, qb);
        const uint32_t pb0 = movmatrix_trans(pack_f16x2(y0.x, y0.y));
        const uint32_t pb1 = movmatrix_trans(pack_f16x2(y1.x, y1.y));
        // zp * 16^b of tokens n and n + 8 as exact fp32 integers (the nibble in place, 2^23 bias off)
        const float2 zz = __fadd2_rn(make_float2(__uint_as_float(0x4B000000u | (zn & (0xFu << (4 * b)))),
                                                 __uint_as_float(0x4B000000u | (zn8 & (0xFu << (4 * b))))),
                                     bc2(-8388608.f));
        float2 z2 = __ffma2_rn(qb, bc2(zz.y), make_float2(zc[b][0], zc[b][1]));
        z2 = __ffma2_rn(qa, bc2(zz.x), z2);
        zc[b][0] = z2.x;
        zc[b][1] = z2.y;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t w01 = vw[b][0] >> (8 * h), w89 = vw[b][1] >> (8 * h);
          mma_f16_16816(o[0][2 * b + h], w01 & kLoNib, w01 & kHiNib, w89 & kLoNib, w89 & kHiNib, pb0, pb1);
        }
      }
      return;
    }
    // zero points of the lane's V^T columns: tokens (2c, 2c+1) and (2c+8, 2c+9)
    // in the two 16-bit halves
    const uint32_t zv01 = lds_u32(vz + 4 * c), zv89 = lds_u32(vz + 4 * c + 16);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float sca = b == 0 ? va01.x : b == 1 ? va01.y : b == 2 ? va23.x : va23.y;
      const float scb = b == 0 ? vb01.x : b == 1 ? vb01.y : b == 2 ? vb23.x : vb23.y;
      uint32_t ph0[NG], ph1[NG], pl0[NG], pl1[NG];
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        // columns (2c, 2c + 1) of tokens n and n + 8 as packed pairs
        const float2 qa = __fmul2_rn(make_float2(pa[g][0], pa[g][1]), bc2(sca));
        const float2 qb = __fmul2_rn(make_float2(pa[g][2], pa[g][3]), bc2(scb));
        const uint32_t h0 = pack_f16x2(qa.x, qa.y), h1 = pack_f16x2(qb.x, qb.y);
        const float2 r0 = __ffma2_rn(half2_bits_to_float2(h0), bc2(-1.f), qa);  // what hi leaves
        const float2 r1 = __ffma2_rn(half2_bits_to_float2(h1), bc2(-1.f), qb);
        ph0[g] = movmatrix_trans(h0);
        ph1[g] = movmatrix_trans(h1);
        pl0[g] = movmatrix_trans(pack_f16x2(r0.x, r0.y));
        pl1[g] = movmatrix_trans(pack_f16x2(r1.x, r1.y));
      }
      // zp as fp16 subnormals in the A layout: rows n (x1) and n + 8 (x16)
      const uint32_t t01 = zv01 >> (4 * b), t89 = zv89 >> (4 * b);
      const uint32_t zl01 = t01 & kLoNib, zh01 = (t01 << 4) & kHiNib;
      const uint32_t zl89 = t89 & kLoNib, zh89 = (t89 << 4) & kHiNib;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t w01 = vw[b][0] >> (8 * h), w89 = vw[b][1] >> (8 * h);
        const uint32_t a0 = hsub2_f16(w01 & kLoNib, zl01), a1 = hsub2_f16(w01 & kHiNib, zh01);
        const uint32_t a2 = hsub2_f16(w89 & kLoNib, zl89), a3 = hsub2_f16(w89 & kHiNib, zh89);
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          mma_f16_16816(o[g][2 * b + h], a0, a1, a2, a3, ph0[g], ph1[g]);
          mma_f16_16816(o[g][2 * b + h], a0, a1, a2, a3, pl0[g], pl1[g]);
        }
      }
    }
  };

  // The token being appended (if this CTA's range holds it): attended from
  // new_kv uncompressed as one more merge state (formed here, before the
  // tiles, so its loads overlap theirs), and quantized into the cache after
  // every tile is consumed. A chunked step: the chunk's tokens, causally, as
  // one more state per column group.
  const int cur = p.cur_from_new ? w.hi - 1 : -1;
  const bool has_cur = w.valid && cur >= w.t_begin && cur < w.t_end;
  if (has_cur && warp == 0) {
    if (CHUNK) {
      // column j of group g (query token ti = slice_first + j / G of slice
      // zs0 + g, head j % G) attends the chunk's tokens 0 .. ti within its
      // window, uncompressed: (m, l, o) of that softmax as its extra state
      const int nq = p.nq;
      const size_t kv_row = ((size_t)w.b * p.kv_heads + w.g) * nq;
      const uint16_t* nk = reinterpret_cast<const uint16_t*>(p.new_kv) + kv_row * 128;
      const uint16_t* nv = reinterpret_cast<const uint16_t*>(p.new_kv) +
                           ((size_t)p.batch * p.kv_heads * nq + kv_row) * 128;
      for (int g = 0; g < nsl; ++g) {
        const int zs = zs0 + g, ncols = G * slice_tokens(p, zs);
        float* xo = extra_o + g * 8 * kOStride;
        for (int j = 0; j < 8; ++j) {
          float mj = -INFINITY, lj = 0.f, o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
          if (j < ncols) {
            const int ti = slice_first(p, zs) + j / G, h = j % G;
            const uint16_t* qj = reinterpret_cast<const uint16_t*>(p.q) +
                                 (((size_t)w.b * p.q_heads + (size_t)w.g * G + h) * nq + ti) * 128;
            const uint2 qq = *reinterpret_cast<const uint2*>(qj + 4 * lane);
            const float q0 = __uint_as_float(qq.x << 16), q1 = __uint_as_float(qq.x & 0xffff0000u);
            const float q2 = __uint_as_float(qq.y << 16), q3 = __uint_as_float(qq.y & 0xffff0000u);
            const int t_first = p.window_q < 0 ? 0 : max(0, ti - p.window_q);
            for (int t = t_first; t <= ti; ++t) {
              const uint2 kk = *reinterpret_cast<const uint2*>(nk + (size_t)t * 128 + 4 * lane);
              float acc = q0 * __uint_as_float(kk.x << 16) + q1 * __uint_as_float(kk.x & 0xffff0000u) +
                          q2 * __uint_as_float(kk.y << 16) + q3 * __uint_as_float(kk.y & 0xffff0000u);
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
              const float st = acc * p.scale_log2;
              const float mn = fmaxf(mj, st);
              const float al = fast_exp2(mj - mn), pt = fast_exp2(st - mn);
              const uint2 vv = *reinterpret_cast<const uint2*>(nv + (size_t)t * 128 + 4 * lane);
              lj = lj * al + pt;
              o0 = o0 * al + pt * __uint_as_float(vv.x << 16);
              o1 = o1 * al + pt * __uint_as_float(vv.x & 0xffff0000u);
              o2 = o2 * al + pt * __uint_as_float(vv.y << 16);
              o3 = o3 * al + pt * __uint_as_float(vv.y & 0xffff0000u);
              mj = mn;
            }
          }
          xo[j * kOStride + 4 * lane + 0] = o0;
          xo[j * kOStride + 4 * lane + 1] = o1;
          xo[j * kOStride + 4 * lane + 2] = o2;
          xo[j * kOStride + 4 * lane + 3] = o3;
          if (lane == 0) {
            ms.wm[(NWARPS + g) * 8 + j] = mj;
            ms.wl[(NWARPS + g) * 8 + j] = lj;
          }
        }
      }
    } else {
      const uint16_t* nk = reinterpret_cast<const uint16_t*>(p.new_kv) + ((size_t)w.b * p.kv_heads + w.g) * 128;
      const uint16_t* nv =
          reinterpret_cast<const uint16_t*>(p.new_kv) + (((size_t)p.batch + w.b) * p.kv_heads + w.g) * 128;
      const uint2 kk = *reinterpret_cast<const uint2*>(nk + 4 * lane);
      const uint2 vv = *reinterpret_cast<const uint2*>(nv + 4 * lane);
      const float k0 = __uint_as_float(kk.x << 16), k1 = __uint_as_float(kk.x & 0xffff0000u);
      const float k2 = __uint_as_float(kk.y << 16), k3 = __uint_as_float(kk.y & 0xffff0000u);
      for (int j = 0; j < 8; ++j) {
        float sj = -INFINITY;
        if (j < G) {
          const uint16_t* qj =
              reinterpret_cast<const uint16_t*>(p.q) + ((size_t)w.b * p.q_heads + (size_t)w.g * G + j) * 128;
          const uint2 qq = *reinterpret_cast<const uint2*>(qj + 4 * lane);
          float acc = __uint_as_float(qq.x << 16) * k0 + __uint_as_float(qq.x & 0xffff0000u) * k1 +
                      __uint_as_float(qq.y << 16) * k2 + __uint_as_float(qq.y & 0xffff0000u) * k3;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
          sj = acc * p.scale_log2;
          extra_o[j * kOStride + 4 * lane + 0] = __uint_as_float(vv.x << 16);
          extra_o[j * kOStride + 4 * lane + 1] = __uint_as_float(vv.x & 0xffff0000u);
          extra_o[j * kOStride + 4 * lane + 2] = __uint_as_float(vv.y << 16);
          extra_o[j * kOStride + 4 * lane + 3] = __uint_as_float(vv.y & 0xffff0000u);
        }
        if (lane == 0) {
          ms.wm[NWARPS * 8 + j] = sj;
          ms.wl[NWARPS * 8 + j] = j < G ? 1.f : 0.f;
        }
      }
    }
  }
  for (int j = 0; j < nstage; ++j) {
    const int tile_idx = j * NWARPS + warp;
    if (tile_idx >= nsub) break;  // the last stage may hold fewer tiles
    const uint32_t jj = (uint32_t)(jbase + j);
    const int st = (int)(jj % STAGES);
    if (!mbar_wait_bounded(bar0 + 8 * st, (jj / STAGES) & 1)) {
      if (lane == 0) set_status(p.status, OL_DEVICE_GUARD);
      break;
    }
    const int t0 = w.t_begin + tile_idx * kTok;
    const uint32_t sg = smem_u32(stages + st * S::kBytes);
    if (t0 >= lo_full && t0 + kTok <= t_stop)
      tile(sg, t0, std::true_type{});
    else
      tile(sg, t0, std::false_type{});
    if (j + STAGES < nstage) {  // every warp has a tile in this stage
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();  // this warp's reads of the stage come first
        if (atomicAdd(freed + st, 1) == NWARPS - 1) {
          freed[st] = 0;
          fence_proxy_async_smem();  // the generic reads before the async-proxy refill
          issue(j + STAGES);
        }
      }
    }
  }
  __syncthreads();  // all stages consumed: they now hold the warps' states

  if constexpr (DUP) {
    // the zero-point term, summed over the tile rows (lanes n), off every dim
    // of its block on the hi lanes (units of O: 2^-24, 16^-b; 16 times more
    // on the rows of upper-nibble dims); then the lo columns added in
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        float v = zc[b][k];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        zc[b][k] = c < 2 ? v * ldexpf(1.f, -24 - 4 * b) : 0.f;
      }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int b = mt >> 1;
      o[0][mt][0] -= zc[b][0];
      o[0][mt][1] -= zc[b][1];
      o[0][mt][2] -= 16.f * zc[b][0];
      o[0][mt][3] -= 16.f * zc[b][1];
#pragma unroll
      for (int k = 0; k < 4; ++k) o[0][mt][k] += __shfl_xor_sync(0xffffffffu, o[0][mt][k], 2);
    }
  }
  if (ev != kNoExp) {  // O to plain units: 2^(24 - ev), and 1/16 more for the rows of upper-nibble dims
    const float f = ldexpf(1.f, 24 - ev), f16 = f * 0.0625f;
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[g][mt][0] *= f;
        o[g][mt][1] *= f;
        o[g][mt][2] *= f16;
        o[g][mt][3] *= f16;
      }
  }
  if (!CHUNK) {
    store_warp_state<true>(reinterpret_cast<float*>(stages + warp * kStateBytes), ms, warp, o[0], mr[0][0], mr[0][1],
                           lr[0][0], lr[0][1]);

    __syncthreads();  // every tile is consumed: the appended row may be rewritten
    if (has_cur && p.append && warp < 2) {
      const int plane = warp;
      const size_t row = (size_t)(plane == 0 ? rowK0 : rowV0) + cur;
      const uint16_t* src = reinterpret_cast<const uint16_t*>(p.new_kv) +
                            (((size_t)plane * p.batch + w.b) * p.kv_heads + w.g) * 128;
      int4_quantize_row_warp(src, 128, p.quant_mode, p.fixed_scale, p.fixed_zp, p.codes + row * 64,
                             p.scales + row * 4, p.zps + row * 2);
    }
    merge_and_finish(
        p, w, has_cur ? NWARPS + 1 : NWARPS,
        [&](int s) {
          return s < NWARPS ? reinterpret_cast<const float*>(stages + s * kStateBytes)
                            : static_cast<const float*>(extra_o);
        },
        merged, cmerged, ms);
  } else {
    // a chunked step: each column group (slice) merged and finished on its own
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      if (g >= nsl) break;
      if (g > 0) {
        // the previous group's merge is complete everywhere (cluster receive
        // buffers read, states and scratch free) before this one reuses them
        if (CS > 1)
          cluster_sync();
        else
          __syncthreads();
        if (threadIdx.x < 8) {  // this group's extra state in the merge's extra slot
          ms.wm[NWARPS * 8 + threadIdx.x] = ms.wm[(NWARPS + g) * 8 + threadIdx.x];
          ms.wl[NWARPS * 8 + threadIdx.x] = ms.wl[(NWARPS + g) * 8 + threadIdx.x];
        }
      }
      store_warp_state<true>(reinterpret_cast<float*>(stages + warp * kStateBytes), ms, warp, o[g], mr[g][0],
                             mr[g][1], lr[g][0], lr[g][1]);
      merge_and_finish(
          p, w, has_cur ? NWARPS + 1 : NWARPS,
          [&](int s) {
            return s < NWARPS ? reinterpret_cast<const float*>(stages + s * kStateBytes)
                              : static_cast<const float*>(extra_o + g * 8 * kOStride);
          },
          merged, cmerged, ms, zs0 + g);
    }
  }
  jbase += nstage;
  if (!p.streamk || w.next < 0) break;
  next = w.next;
  }  // segments
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

// A [2 planes][rows][inner] byte array as a 3-D tensor map whose boxes span
// `box_rows` rows of both planes.
bool encode_planes(CUtensorMap* map, void* base, uint64_t inner, uint64_t rows, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, rows, 2};
  cuuint64_t strides[2] = {inner, inner * rows};
  cuuint32_t box[3] = {(cuuint32_t)inner, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The three maps of a stage of NWARPS tiles: codes as 64-byte rows, scales as
// 16-byte rows of two tokens, zero points as 16-byte rows of eight tokens.
bool encode_int4_maps(CUtensorMap (&maps)[3], const AttnParams& p, int nwarps) {
  const uint64_t rows = (uint64_t)p.batch * p.kv_heads * p.capacity;  // per plane
  const uint32_t tok = 16u * nwarps;
  return encode_planes(&maps[0], p.codes, 64, rows, tok, CU_TENSOR_MAP_SWIZZLE_64B) &&
         encode_planes(&maps[1], p.scales, 16, rows / 2, tok / 2, CU_TENSOR_MAP_SWIZZLE_NONE) &&
         encode_planes(&maps[2], p.zps, 16, rows / 8, tok / 8, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int NWARPS, int STAGES, bool CHUNK = false, bool DUP = false>
cudaError_t ensure_attrs() {
  static cudaError_t state = [] {
    auto kern = fast_int4_kernel<NWARPS, STAGES, CHUNK, DUP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Int4Layout<NWARPS, STAGES, CHUNK ? 2 : 1>::kTotal);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
  }();
  return state;
}

template <int NWARPS, int STAGES>
int max_cluster() {
  static int cs = [] {
    if (ensure_attrs<NWARPS, STAGES>() != cudaSuccess) return 1;
    for (int c = 16; c >= 2; c >>= 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(c, 1, 1);
      cfg.blockDim = dim3(NWARPS * 32, 1, 1);
      cfg.dynamicSmemBytes = Int4Layout<NWARPS, STAGES>::kTotal;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = c;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, fast_int4_kernel<NWARPS, STAGES>, &cfg) == cudaSuccess && n > 0)
        return c;
      cudaGetLastError();
    }
    return 1;
  }();
  return cs;
}

template <int NWARPS, int STAGES, bool CHUNK, bool DUP = false>
cudaError_t launch_cfg(const AttnParams& p, cudaStream_t s) {
  CUtensorMap maps[3];
  if (!encode_int4_maps(maps, p, NWARPS)) return cudaErrorInvalidValue;
  cudaError_t e = ensure_attrs<NWARPS, STAGES, CHUNK, DUP>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  // a chunked step: pairs of slices of query tokens along x (a CTA carries two
  // slices' columns), the plan's CTAs (and clusters) along y
  const int slices = CHUNK ? (p.nq + p.tq - 1) / p.tq : 1;
  cfg.gridDim = CHUNK ? dim3((slices + 1) / 2, p.total_ctas, 1) : dim3(p.total_ctas, 1, 1);
  cfg.blockDim = dim3(NWARPS * 32, 1, 1);
  cfg.dynamicSmemBytes = Int4Layout<NWARPS, STAGES, CHUNK ? 2 : 1>::kTotal;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CHUNK ? 1 : p.cluster;
  attr[1].val.clusterDim.y = CHUNK ? p.cluster : 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fast_int4_kernel<NWARPS, STAGES, CHUNK, DUP>, maps[0], maps[1], maps[2], p);
}

}  // namespace

bool fast_int4_supported(const AttnParams& p) {
  if (p.layout != OL_LAYOUT_INT4 || p.head_dim != 128 || p.group > 8) return false;
  // a chunked step: query tokens share a CTA as extra columns (at most 8)
  if (p.nq > 1 && (p.tq < 1 || p.group * p.tq > 8)) return false;
  // every (row, kv head) starts on a 16-token boundary, so a stage's scale
  // and zero-point boxes start on whole 16-byte rows of their maps
  if (p.capacity % 16 != 0) return false;
  const unsigned long long rows = 2ull * p.batch * p.kv_heads * p.capacity;
  return rows < (1ull << 31);
}

int fast_int4_smem(int variant) {
  switch (variant) {
    case 1: return Int4Layout<4, 4>::kTotal;
    case 2: return Int4Layout<8, 2>::kTotal;
    default: return Int4Layout<6, 6>::kTotal;
  }
}
// variant 0 (the default): decode steps 6 warps x 6 stages, two CTAs per SM at
// up to 168 registers (int4_b16 88.2 us/step; 4 stages 89.2, 8 warps x 4 at
// 128 registers 91.6); chunked steps keep 8 warps x 4 stages (two column
// groups, one CTA per SM)
int fast_int4_warps(int variant) { return variant == 1 ? 4 : variant == 0 ? 6 : 8; }
int fast_int4_ctas_per_sm(int variant, bool chunk) {
  switch (variant) {
    case 1: return chunk ? Int4Layout<4, 4, 2>::kPerSm : Int4Layout<4, 4>::kPerSm;
    case 2: return chunk ? Int4Layout<8, 2, 2>::kPerSm : Int4Layout<8, 2>::kPerSm;
    default: return chunk ? Int4Layout<8, 4, 2>::kPerSm : Int4Layout<6, 6>::kPerSm;
  }
}
int fast_int4_max_cluster(int variant) {
  switch (variant) {
    case 1: return max_cluster<4, 4>();
    case 2: return max_cluster<8, 2>();
    default: return max_cluster<6, 6>();
  }
}

cudaError_t launch_fast_int4(const AttnParams& p, cudaStream_t s) {
  if (p.total_ctas <= 0) return cudaSuccess;
  if (p.nq > 1) {
    switch (p.variant) {
      case 1: return launch_cfg<4, 4, true>(p, s);
      case 2: return launch_cfg<8, 2, true>(p, s);
      default: return launch_cfg<8, 4, true>(p, s);
    }
  }
  if (p.group <= 4) {  // the lo half of P^T in the free MMA columns
    switch (p.variant) {
      case 1: return launch_cfg<4, 4, false, true>(p, s);
      case 2: return launch_cfg<8, 2, false, true>(p, s);
      default: return launch_cfg<6, 6, false, true>(p, s);
    }
  }
  switch (p.variant) {
    case 1: return launch_cfg<4, 4, false>(p, s);
    case 2: return launch_cfg<8, 2, false>(p, s);
    default: return launch_cfg<6, 6, false>(p, s);
  }
}

}  // namespace ol
