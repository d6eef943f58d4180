// ol_fast_int4.cu -- tensor-core decode attention (and fused quantize-append)
// over the INT4 blockwise-affine cache with head_dim 128 and a GQA group of at
// most 8: codes [2, B, Hkv, C, 64] (two uint4 per byte, low nibble first),
// fp16 scales [2, B, Hkv, C, 4] and zero points [2, B, Hkv, C, 2] (two uint4
// per byte), one (scale, zero point) per block of 32 dims.
//
// Same decomposition as the bf16 kernel (one CTA per (row, kv head, split),
// per-warp rings of 16-token tiles, shared merge). Per tile a warp receives
// 2 x 1 KB of codes by TMA (SWIZZLE_64B, 64-byte rows: conflict-free reads)
// and 2 x 128 B of scales and 2 x 32 B of zero points by bulk copies.
// Dequantization happens in registers: a nibble c becomes the exact bf16
// value 128 + c with one mask-and-or per pair.
//   S^T: one accumulator per 32-dim block b, fed the exact bf16 values
//        (128 + c) - (128 + zp_K) = c - zp_K; then s = sum_b scale_K[t,b] * acc_b
//   O^T: V^T as exact bf16 (c - zp_V) per token, the V scale folded into
//        P^T per block, P^T carried as bf16 hi + lo.
// The token being appended (fused step) takes part uncompressed from new_kv as
// one extra merge state, and is quantized into the cache by the same CTA.
#include <cuda_bf16.h>

#include "ol_merge.cuh"

namespace ol {
namespace {

constexpr int kTok = 16;
constexpr int kCodesBytes = kTok * 64;    // one plane's codes of a tile
constexpr int kScaleBytes = kTok * 8;     // 4 fp16 per row
constexpr int kZpBytes = kTok * 2;        // 4 nibbles per row
constexpr int kTileTx = 2 * (kCodesBytes + kScaleBytes + kZpBytes);  // 2368
constexpr int kStage = 3072;              // 1024-aligned stage stride
constexpr int kOffVc = 1024, kOffSk = 2048, kOffSv = 2048 + 128, kOffZk = 2304, kOffZv = 2336;
constexpr uint32_t kMagic = 0x43004300u;  // bf16 pair (128, 128)

template <int NWARPS, int STAGES>
struct Int4Layout {
  static constexpr int kStages = NWARPS * STAGES * kStage;
  // extra state O, then one region that is either the CTA-merged state (no
  // cluster) or the cluster receive buffers + cmerged (cluster): never both
  static constexpr int kUnion = (1024 + 2 * 128 + 8 * 64) * 4 > 8 * kOStride * 4 ? (1024 + 2 * 128 + 8 * 64) * 4
                                                                               : 8 * kOStride * 4;
  static constexpr int kExtra = 8 * kOStride * 4 + kUnion;
  static constexpr int kBars = NWARPS * STAGES * 8;
  static constexpr int kMisc = 256 + (NWARPS + 1) * 8 * 4 * 2 + 8 * 4 * 6 + 16 * 4 + 2 * 16 * 8 * 4 + 16;
  static constexpr int kTotal = 1024 + kStages + kExtra + kBars + kMisc;
  static constexpr int kPerSm = (228 * 1024) / (kTotal + 1024) > 0 ? (228 * 1024) / (kTotal + 1024) : 1;
  static_assert(STAGES * kStage >= 8 * kOStride * 4, "a warp's state fits its stages");
};

__device__ __forceinline__ uint32_t code_pair(uint32_t w, int shift) {
  return ((w >> shift) & 0x000F000Fu) | kMagic;
}
__device__ __forceinline__ uint32_t hsub2_bf16(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a), y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 r = __hsub2(x, y);
  return *reinterpret_cast<uint32_t*>(&r);
}
// byte offset of logical byte x of 64-byte row r in a SWIZZLE_64B tile
__device__ __forceinline__ int swz64(int r, int x) {
  return r * 64 + ((((x >> 4) ^ (r >> 1)) & 3) << 4) + (x & 15);
}

template <int NWARPS, int STAGES>
__global__ void __launch_bounds__(NWARPS * 32, Int4Layout<NWARPS, STAGES>::kPerSm)
    fast_int4_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ AttnParams p) {
  using L = Int4Layout<NWARPS, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* stages = smem;
  float* extra_o = reinterpret_cast<float*>(smem + L::kStages);
  float* merged = extra_o + 8 * kOStride;  // no cluster: the CTA state
  float* recv = merged;                    // cluster: receive buffers, then cmerged
  float* cmerged = recv + 1024 + 256;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kStages + L::kExtra);
  Work* sw = reinterpret_cast<Work*>(smem + L::kStages + L::kExtra + L::kBars);
  float* misc = reinterpret_cast<float*>(smem + L::kStages + L::kExtra + L::kBars + 256);
  MergeScratch ms;
  ms.wm = misc;                        // [NWARPS + 1][8]
  ms.wl = ms.wm + (NWARPS + 1) * 8;    // [NWARPS + 1][8]
  ms.m = ms.wl + (NWARPS + 1) * 8;
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
  if (threadIdx.x == 0) prefetch_tensormap(&tmap);
  const uint32_t bar0 = smem_u32(bars + warp * STAGES);
  if (lane == 0) {
    for (int st = 0; st < STAGES; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_mbar_init();
  }
  if (!p.inline_lens) pdl_wait();
  if (warp == 0) {
    Work w = p.inline_lens
                 ? map_cta_warp(p.lens_inline, p.batch, p.kv_heads, p.capacity, p.window, p.chunk, blockIdx.x,
                                nullptr, CS)
                 : map_cta_warp(p.lens, p.batch, p.kv_heads, p.capacity, p.window, p.chunk, blockIdx.x, p.status, CS);
    if (lane == 0) *sw = w;
  }
  __syncthreads();
  const Work w = *sw;
  if (!w.valid && CS == 1) {
    if (p.inline_lens) pdl_wait();
    return;
  }

  const int G = p.group;
  const int C = p.capacity;
  const int nsub = w.valid ? (w.t_end - w.t_begin + kTok - 1) / kTok : 0;
  const int my_n = nsub > warp ? (nsub - warp + NWARPS - 1) / NWARPS : 0;
  uint8_t* my_stages = stages + warp * STAGES * kStage;
  const uint64_t pol = policy_evict_first();
  const int rowK0 = ((0 * p.batch + w.b) * p.kv_heads + w.g) * C;  // row of token 0, K plane
  const int rowV0 = ((1 * p.batch + w.b) * p.kv_heads + w.g) * C;

  auto issue = [&](int i) {
    const int st = i % STAGES;
    const int t0 = w.t_begin + (warp + i * NWARPS) * kTok;
    uint8_t* dst = my_stages + st * kStage;
    const uint32_t bar = bar0 + 8 * st;
    mbar_arrive_expect_tx(bar, kTileTx);
    tma_load_2d(smem_u32(dst), &tmap, 0, rowK0 + t0, bar, pol);
    tma_load_2d(smem_u32(dst + kOffVc), &tmap, 0, rowV0 + t0, bar, pol);
    bulk_load(smem_u32(dst + kOffSk), p.scales + (size_t)(rowK0 + t0) * 4, kScaleBytes, bar, pol);
    bulk_load(smem_u32(dst + kOffSv), p.scales + (size_t)(rowV0 + t0) * 4, kScaleBytes, bar, pol);
    bulk_load(smem_u32(dst + kOffZk), p.zps + (size_t)(rowK0 + t0) * 2, kZpBytes, bar, pol);
    bulk_load(smem_u32(dst + kOffZv), p.zps + (size_t)(rowV0 + t0) * 2, kZpBytes, bar, pol);
  };
  const int pre = my_n < STAGES ? my_n : STAGES;
  if (p.early && lane == 0)
    for (int i = 0; i < pre; ++i) issue(i);
  if (p.inline_lens) pdl_wait();
  pdl_launch_dependents();
  if (!p.early && lane == 0)
    for (int i = 0; i < pre; ++i) issue(i);

  // q as the B operand of the four blocks' k-steps, in the dims order of the
  // code words: lane (c, n) holds q[n][32b + 8c .. +7] as e0..e7;
  // k-step (b, hh): b0 = {e(2hh), e(2hh+4)}, b1 = {e(2hh+1), e(2hh+5)}.
  const int c = lane & 3, n = lane >> 2;
  uint32_t qf[4][2][2];
  {
    const bool live = n < G && w.valid;
    const uint16_t* qp = reinterpret_cast<const uint16_t*>(p.q) +
                         ((size_t)w.b * p.q_heads + (size_t)w.g * G + (n < G ? n : 0)) * 128;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      uint4 v = live ? __ldg(reinterpret_cast<const uint4*>(qp + 32 * b + 8 * c)) : make_uint4(0, 0, 0, 0);
      qf[b][0][0] = __byte_perm(v.x, v.z, 0x5410);
      qf[b][0][1] = __byte_perm(v.x, v.z, 0x7632);
      qf[b][1][0] = __byte_perm(v.y, v.w, 0x5410);
      qf[b][1][1] = __byte_perm(v.y, v.w, 0x7632);
    }
  }
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m_run0 = -INFINITY, m_run1 = -INFINITY, l_run0 = 0.f, l_run1 = 0.f;
  const int codes_hi = p.cur_from_new ? w.hi - 1 : w.hi;  // tokens below this come from the codes
  const int t_stop = min(w.t_end, codes_hi);

  for (int i = 0; i < my_n; ++i) {
    const int st = i % STAGES;
    if (!mbar_wait_bounded(bar0 + 8 * st, (i / STAGES) & 1)) {
      if (lane == 0) set_status(p.status, OL_DEVICE_GUARD);
      break;
    }
    const int t0 = w.t_begin + (warp + i * NWARPS) * kTok;
    const uint32_t sg = smem_u32(my_stages + st * kStage);
    const uint32_t kc = sg, vc = sg + kOffVc, ksc = sg + kOffSk, vsc = sg + kOffSv, kz = sg + kOffZk, vz = sg + kOffZv;

    const int ra = n, rb = n + 8;  // the lane's S^T rows (tokens) in this tile
    const bool va = t0 + ra >= w.lo && t0 + ra < t_stop;
    const bool vb = t0 + rb >= w.lo && t0 + rb < t_stop;

    // ---- S^T = K q^T, one accumulator per 32-dim block, A = exact (c - zp)
    // zero points of rows ra / rb, duplicated in both 16-bit halves
    const uint32_t za = lds_u16(kz + 2 * ra), zb = lds_u16(kz + 2 * rb);
    const uint32_t zda = za | (za << 16), zdb = zb | (zb << 16);
    float sacc[4][4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      sacc[b][0] = sacc[b][1] = sacc[b][2] = sacc[b][3] = 0.f;
      const uint32_t wa = lds_u32(kc + swz64(ra, 16 * b + 4 * c));
      const uint32_t wb = lds_u32(kc + swz64(rb, 16 * b + 4 * c));
      const uint32_t zpa = code_pair(zda, 4 * b), zpb = code_pair(zdb, 4 * b);  // (128 + zp, 128 + zp)
      mma_bf16_16816(sacc[b], hsub2_bf16(code_pair(wa, 0), zpa), hsub2_bf16(code_pair(wb, 0), zpb),
                     hsub2_bf16(code_pair(wa, 4), zpa), hsub2_bf16(code_pair(wb, 4), zpb), qf[b][0][0],
                     qf[b][0][1]);
      mma_bf16_16816(sacc[b], hsub2_bf16(code_pair(wa, 8), zpa), hsub2_bf16(code_pair(wb, 8), zpb),
                     hsub2_bf16(code_pair(wa, 12), zpa), hsub2_bf16(code_pair(wb, 12), zpb), qf[b][1][0],
                     qf[b][1][1]);
    }
    const uint2 ska = lds_v2(ksc + 8 * ra);
    const uint2 skb = lds_v2(ksc + 8 * rb);
    float s00 = 0.f, s01 = 0.f, s10 = 0.f, s11 = 0.f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t pa = b < 2 ? ska.x : ska.y, pb = b < 2 ? skb.x : skb.y;
      const float sca = fp16_bits_to_float((b & 1) ? (pa >> 16) : (pa & 0xffff));
      const float scb = fp16_bits_to_float((b & 1) ? (pb >> 16) : (pb & 0xffff));
      s00 += sca * sacc[b][0];
      s01 += sca * sacc[b][1];
      s10 += scb * sacc[b][2];
      s11 += scb * sacc[b][3];
    }
    s00 = va ? s00 * p.scale_log2 : -INFINITY;
    s01 = va ? s01 * p.scale_log2 : -INFINITY;
    s10 = vb ? s10 * p.scale_log2 : -INFINITY;
    s11 = vb ? s11 * p.scale_log2 : -INFINITY;

    // ---- online softmax (exp2 domain)
    float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m_run0, mx0), mn1 = fmaxf(m_run1, mx1);
    const float b0 = mn0 == -INFINITY ? 0.f : mn0, b1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = fast_exp2(m_run0 - b0), al1 = fast_exp2(m_run1 - b1);
    const float p00 = fast_exp2(s00 - b0), p01 = fast_exp2(s01 - b1);
    const float p10 = fast_exp2(s10 - b0), p11 = fast_exp2(s11 - b1);
    l_run0 = l_run0 * al0 + (p00 + p10);
    l_run1 = l_run1 * al1 + (p01 + p11);
    // rescale O only when some lane's running maximum moved (otherwise every
    // factor is exactly 1)
    if (__any_sync(0xffffffffu, mn0 != m_run0 || mn1 != m_run1)) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= al0;
        o[mt][1] *= al1;
        o[mt][2] *= al0;
        o[mt][3] *= al1;
      }
    }
    m_run0 = mn0;
    m_run1 = mn1;

    // ---- O^T += V^T P^T, block by block
    const uint2 sva = lds_v2(vsc + 8 * ra);
    const uint2 svb = lds_v2(vsc + 8 * rb);
    const int r0 = 2 * c, r1 = 2 * c + 1, r8 = 2 * c + 8, r9 = 2 * c + 9;  // V^T columns (tokens) of this lane
    // zero points of those tokens: tokens (r0, r1) in the two 16-bit halves, likewise (r8, r9)
    const uint32_t zv01 = lds_u16(vz + 2 * r0) | (lds_u16(vz + 2 * r1) << 16);
    const uint32_t zv89 = lds_u16(vz + 2 * r8) | (lds_u16(vz + 2 * r9) << 16);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t pa = b < 2 ? sva.x : sva.y, pb = b < 2 ? svb.x : svb.y;
      const float sca = va ? fp16_bits_to_float((b & 1) ? (pa >> 16) : (pa & 0xffff)) : 0.f;
      const float scb = vb ? fp16_bits_to_float((b & 1) ? (pb >> 16) : (pb & 0xffff)) : 0.f;
      const float q00 = p00 * sca, q01 = p01 * sca, q10 = p10 * scb, q11 = p11 * scb;
      const uint32_t h0 = pack_bf16x2(q00, q01), h1 = pack_bf16x2(q10, q11);
      const uint32_t l0 = pack_bf16x2(q00 - __uint_as_float(h0 << 16), q01 - __uint_as_float(h0 & 0xffff0000u));
      const uint32_t l1 = pack_bf16x2(q10 - __uint_as_float(h1 << 16), q11 - __uint_as_float(h1 & 0xffff0000u));
      const uint32_t ph0 = movmatrix_trans(h0), ph1 = movmatrix_trans(h1);
      const uint32_t pl0 = movmatrix_trans(l0), pl1 = movmatrix_trans(l1);
      // V codes of this lane's dims (32b + 4n .. +3) for tokens r0, r1, r8, r9
      const int x = 16 * b + 2 * n;
      const uint32_t w01 = lds_u16(vc + swz64(r0, x)) | (lds_u16(vc + swz64(r1, x)) << 16);
      const uint32_t w89 = lds_u16(vc + swz64(r8, x)) | (lds_u16(vc + swz64(r9, x)) << 16);
      const uint32_t z01 = code_pair(zv01, 4 * b), z89 = code_pair(zv89, 4 * b);  // (128 + zp) per token
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t a0 = hsub2_bf16(code_pair(w01, 8 * h), z01);
        const uint32_t a1 = hsub2_bf16(code_pair(w01, 8 * h + 4), z01);
        const uint32_t a2 = hsub2_bf16(code_pair(w89, 8 * h), z89);
        const uint32_t a3 = hsub2_bf16(code_pair(w89, 8 * h + 4), z89);
        mma_bf16_16816(o[2 * b + h], a0, a1, a2, a3, ph0, ph1);
        mma_bf16_16816(o[2 * b + h], a0, a1, a2, a3, pl0, pl1);
      }
    }
    __syncwarp();
    if (lane == 0 && i + STAGES < my_n) {
      fence_proxy_async_smem();  // this stage's generic reads before the async-proxy refill
      issue(i + STAGES);
    }
  }

  store_warp_state<true>(reinterpret_cast<float*>(my_stages), ms, warp, o, m_run0, m_run1, l_run0, l_run1);

  // The token being appended (if this CTA's range holds it): attended from
  // new_kv uncompressed as one more merge state, and quantized into the cache.
  const int cur = p.cur_from_new ? w.hi - 1 : -1;
  const bool has_cur = w.valid && cur >= w.t_begin && cur < w.t_end;
  if (has_cur && warp == 0) {
    const uint16_t* nk = reinterpret_cast<const uint16_t*>(p.new_kv) + ((size_t)w.b * p.kv_heads + w.g) * 128;
    const uint16_t* nv = reinterpret_cast<const uint16_t*>(p.new_kv) + (((size_t)p.batch + w.b) * p.kv_heads + w.g) * 128;
    const uint2 kk = *reinterpret_cast<const uint2*>(nk + 4 * lane);
    const uint2 vv = *reinterpret_cast<const uint2*>(nv + 4 * lane);
    const float k0 = __uint_as_float(kk.x << 16), k1 = __uint_as_float(kk.x & 0xffff0000u);
    const float k2 = __uint_as_float(kk.y << 16), k3 = __uint_as_float(kk.y & 0xffff0000u);
    for (int j = 0; j < 8; ++j) {
      float sj = -INFINITY;
      if (j < G) {
        const uint16_t* qj = reinterpret_cast<const uint16_t*>(p.q) + ((size_t)w.b * p.q_heads + (size_t)w.g * G + j) * 128;
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
  __syncthreads();  // every warp's tiles are consumed: the appended row may be rewritten
  if (has_cur && p.append && warp < 2) {
    const int plane = warp;
    const size_t row = (size_t)(plane == 0 ? rowK0 : rowV0) + cur;
    const uint16_t* src = reinterpret_cast<const uint16_t*>(p.new_kv) +
                          (((size_t)plane * p.batch + w.b) * p.kv_heads + w.g) * 128;
    int4_quantize_row_warp(src, 128, p.quant_mode, p.fixed_scale, p.fixed_zp, p.codes + row * 64, p.scales + row * 4,
                           p.zps + row * 2);
  }
  merge_and_finish(
      p, w, has_cur ? NWARPS + 1 : NWARPS,
      [&](int s) {
        return s < NWARPS ? reinterpret_cast<const float*>(stages + s * STAGES * kStage)
                          : static_cast<const float*>(extra_o);
      },
      merged, cmerged, ms);
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

// codes plane as rows of 64 bytes; boxes of 16 rows, 64-byte swizzle
bool encode_codes(CUtensorMap* map, void* base, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {64, rows};
  cuuint64_t strides[1] = {64};
  cuuint32_t box[2] = {64, kTok};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NWARPS, int STAGES>
cudaError_t ensure_attrs() {
  static cudaError_t state = [] {
    auto kern = fast_int4_kernel<NWARPS, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Int4Layout<NWARPS, STAGES>::kTotal);
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

template <int NWARPS, int STAGES>
cudaError_t launch_cfg(const CUtensorMap& map, const AttnParams& p, cudaStream_t s) {
  cudaError_t e = ensure_attrs<NWARPS, STAGES>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.total_ctas, 1, 1);
  cfg.blockDim = dim3(NWARPS * 32, 1, 1);
  cfg.dynamicSmemBytes = Int4Layout<NWARPS, STAGES>::kTotal;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = p.cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fast_int4_kernel<NWARPS, STAGES>, map, p);
}

}  // namespace

bool fast_int4_supported(const AttnParams& p) {
  if (p.layout != OL_LAYOUT_INT4 || p.head_dim != 128 || p.group > 8) return false;
  // tiles never cross a row's capacity (the bulk copies of scales and zero
  // points have no out-of-bounds fill) and start 16-byte aligned
  if (p.capacity % 16 != 0) return false;
  const unsigned long long rows = 2ull * p.batch * p.kv_heads * p.capacity;
  return rows < (1ull << 31);
}

int fast_int4_smem(int variant) {
  switch (variant) {
    case 1: return Int4Layout<4, 4>::kTotal;
    case 2: return Int4Layout<8, 2>::kTotal;
    default: return Int4Layout<8, 4>::kTotal;
  }
}
int fast_int4_warps(int variant) { return variant == 1 ? 4 : 8; }
int fast_int4_max_cluster(int variant) {
  switch (variant) {
    case 1: return max_cluster<4, 4>();
    case 2: return max_cluster<8, 2>();
    default: return max_cluster<8, 4>();
  }
}

cudaError_t launch_fast_int4(const AttnParams& p, cudaStream_t s) {
  if (p.total_ctas <= 0) return cudaSuccess;
  CUtensorMap map;
  if (!encode_codes(&map, p.codes, 2ull * p.batch * p.kv_heads * p.capacity)) return cudaErrorInvalidValue;
  switch (p.variant) {
    case 1: return launch_cfg<4, 4>(map, p, s);
    case 2: return launch_cfg<8, 2>(map, p, s);
    default: return launch_cfg<8, 4>(map, p, s);
  }
}

}  // namespace ol
