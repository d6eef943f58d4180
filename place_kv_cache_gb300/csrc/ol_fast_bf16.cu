// ol_fast_bf16.cu -- tensor-core decode attention (and fused append) for bf16
// caches with head_dim 128 and a GQA group of at most 8 query heads, over the
// contiguous cache [2, B, Hkv, C, 128] or the paged pool [2, P, Hkv, S, 128]
// (S a multiple of 16).
//
// Work decomposition: one CTA per (row, kv head, split of `chunk` tokens);
// every byte of K/V is read once, by the CTA that serves the whole GQA group.
// Inside the CTA each warp owns the 16-token tiles w, w + NWARPS, ... of the
// split and runs its own STAGES-deep ring: TMA 2D tensor copies (SWIZZLE_128B,
// 64-dim halves of 16 rows) land K and V tiles in shared memory, completion
// on one mbarrier per stage.
//
// Per tile, with the group's q as the N = 8 side of m16n8k16 (GQA <= 8 forms a
// real dense 16x8 tile; padding heads carry q = 0):
//   S^T[16 tok x 8 heads] = K[16 x 128] * q^T        8 mma, K via ldmatrix
//   online softmax on S^T columns (exp2 domain, fp32)
//   P^T (bf16) from the S^T accumulator by movmatrix.trans
//   O^T[128 dims x 8 heads] += V^T[128 x 16] * P^T  8 mma, V via ldmatrix.trans
// Warps merge in shared memory; CTAs of one (row, kv head) merge through
// fp32 partials in the workspace and an atomic ticket (finish_split).
#include "ol_merge.cuh"

namespace ol {
namespace {

constexpr int kTok = 16;                    // tokens per tile
constexpr int kHalfBytes = kTok * 128;      // 16 rows x 64 bf16 (one SWIZZLE_128B box)
constexpr int kPlaneBytes = 2 * kHalfBytes; // K or V tile: 4 KB
constexpr int kStageBytes = 2 * kPlaneBytes;// K + V: 8 KB

template <int NWARPS, int STAGES>
struct FastLayout {
  static constexpr int kStages = NWARPS * STAGES * kStageBytes;
  static constexpr int kBars = NWARPS * STAGES * 8;
  static constexpr int kMisc = 256 + NWARPS * 8 * 4 * 2 + 8 * 4 * 6 + 2 * 16 * 8 * 4 + 16;
  static constexpr int kRecv = (1024 + 2 * 128 + 8 * 64) * 4;  // cluster receive buffers + cmerged
  static constexpr int kTotal = 1024 /* alignment slack */ + kStages + kRecv + kBars + kMisc;
  // CTAs per SM that shared memory allows (1 KB per CTA is reserved by the driver)
  static constexpr int kPerSm = (228 * 1024) / (kTotal + 1024) > 0 ? (228 * 1024) / (kTotal + 1024) : 1;
  static_assert(STAGES >= 2, "the merged O lives in warp 0's second stage");
  static_assert(8 * kOStride * 4 <= kStageBytes, "the CTA state fits one stage");
};

__device__ __forceinline__ int tile_row(const AttnParams& p, bool paged, int plane, int b, int g, int t0,
                                        bool* bad) {
  if (!paged) return (((plane * p.batch + b) * p.kv_heads + g) * p.capacity) + t0;
  int page = __ldg(p.block_table + (size_t)b * p.max_pages + t0 / p.page_size);
  if (page < 0 || page >= p.num_pages) {
    *bad = true;
    page = 0;
  }
  return ((plane * p.num_pages + page) * p.kv_heads + g) * p.page_size + (t0 % p.page_size);
}

template <int NWARPS, int STAGES, bool PAGED>
__global__ void __launch_bounds__(NWARPS * 32, FastLayout<NWARPS, STAGES>::kPerSm)
    fast_bf16_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ AttnParams p) {
  using L = FastLayout<NWARPS, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* stages = smem;
  float* recv = reinterpret_cast<float*>(smem + L::kStages);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kStages + L::kRecv);
  Work* sw = reinterpret_cast<Work*>(smem + L::kStages + L::kRecv + L::kBars);
  float* misc = reinterpret_cast<float*>(smem + L::kStages + L::kRecv + L::kBars + 256);
  MergeScratch ms;
  ms.wm = misc;                 // [NWARPS][8]
  ms.wl = ms.wm + NWARPS * 8;   // [NWARPS][8]
  ms.m = ms.wl + NWARPS * 8;    // [8]
  ms.l = ms.m + 8;
  ms.cm = ms.l + 8;
  ms.cl = ms.cm + 8;
  ms.scr = ms.cl + 8;           // [16]
  ms.cw = ms.scr + 16;          // [16][8]
  ms.wt = ms.cw + 16 * 8;       // [16][8] (>= nstates x 8)
  ms.flag = reinterpret_cast<int*>(ms.wt + 16 * 8);
  ms.recv_o = recv;             // [1024]
  ms.recv_m = recv + 1024;      // [128]
  ms.recv_l = recv + 1024 + 128;
  float* cmerged = recv + 1024 + 256;  // [8][64]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int CS = p.cluster;
  if (threadIdx.x == 0) prefetch_tensormap(&tmap);
  const uint32_t bar0 = smem_u32(bars + warp * STAGES);
  if (lane == 0) {
    for (int st = 0; st < STAGES; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_mbar_init();
  }
  // With the lengths carried in the launch the CTA mapping needs no memory
  // written by earlier work and runs before the dependency wait; so do the
  // first TMA requests when the caller declared the history stable.
  if (!p.inline_lens) pdl_wait();
  if (warp == 0) {
    Work w = p.inline_lens
                 ? map_cta_warp(p.lens_inline, p.batch, p.kv_heads, p.capacity, p.window, p.chunk, cta_index(p),
                                nullptr, CS)
                 : map_cta_warp(p.lens, p.batch, p.kv_heads, p.capacity, p.window, p.chunk, cta_index(p), p.status,
                                CS);
    slice_query(w, p);
    if (lane == 0) *sw = w;
  }
  __syncthreads();
  const Work w = *sw;
  // Without a cluster an unmapped CTA can leave now; in a cluster every CTA
  // must reach the cluster barriers, so it runs with an empty token range.
  if (!w.valid && CS == 1) {
    if (p.inline_lens) pdl_wait();
    return;
  }

  const int G = p.group;
  const int nsub = w.valid ? (w.t_end - w.t_begin + kTok - 1) / kTok : 0;
  const int my_n = nsub > warp ? (nsub - warp + NWARPS - 1) / NWARPS : 0;
  uint8_t* my_stages = stages + warp * STAGES * kStageBytes;
  // a decode step reads each K/V byte once; a chunk's query tokens re-read it from L2
  const uint64_t pol = p.nq > 1 ? policy_evict_normal() : policy_evict_first();

  // lane 0 issues the four TMA boxes of this warp's i-th tile into stage i % STAGES
  auto issue = [&](int i) {
    const int st = i % STAGES;
    const int t0 = w.t_begin + (warp + i * NWARPS) * kTok;
    bool bad = false;
    const int rk = tile_row(p, PAGED, 0, w.b, w.g, t0, &bad);
    const int rv = tile_row(p, PAGED, 1, w.b, w.g, t0, &bad);
    if (bad) set_status(p.status, OL_DEVICE_GUARD);
    const uint32_t dst = smem_u32(my_stages + st * kStageBytes);
    const uint32_t bar = bar0 + 8 * st;
    mbar_arrive_expect_tx(bar, kStageBytes);
    tma_load_2d(dst, &tmap, 0, rk, bar, pol);
    tma_load_2d(dst + kHalfBytes, &tmap, 64, rk, bar, pol);
    tma_load_2d(dst + kPlaneBytes, &tmap, 0, rv, bar, pol);
    tma_load_2d(dst + kPlaneBytes + kHalfBytes, &tmap, 64, rv, bar, pol);
  };
  const int pre = my_n < STAGES ? my_n : STAGES;
  if (p.early && lane == 0)
    for (int i = 0; i < pre; ++i) issue(i);
  if (p.inline_lens) pdl_wait();
  pdl_launch_dependents();
  if (!p.early && lane == 0)
    for (int i = 0; i < pre; ++i) issue(i);

  // q^T as the B operand (16 dims x 8 heads per k-step): lane (c, n) holds
  // q[n][16kk + 2c, +1] and q[n][16kk + 2c + 8, +9]; heads n >= G are zero.
  const int c = lane & 3, n = lane >> 2;
  uint32_t qf[8][2];
  {
    const uint16_t* qp = reinterpret_cast<const uint16_t*>(p.q) +
                         (((size_t)w.b * p.q_heads + (size_t)w.g * G + (n < G ? n : 0)) * (p.nq > 1 ? p.nq : 1) +
                          query_index(p)) * 128;
    const bool live = n < G && w.valid;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qf[kk][0] = live ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * kk + 2 * c)) : 0u;
      qf[kk][1] = live ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * kk + 2 * c + 8)) : 0u;
    }
  }

  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m_run0 = -INFINITY, m_run1 = -INFINITY, l_run0 = 0.f, l_run1 = 0.f;

  // ldmatrix lane roles: matrix mi = lane / 8, row r8 = lane % 8
  const int mi = lane >> 3, r8 = lane & 7;
  const int rK = r8 + 8 * (mi & 1), cK = mi >> 1;  // K: tokens, dim chunk offset
  const int rV = r8 + 8 * (mi >> 1), cV = mi & 1;  // V (transposed): tokens, dim chunk offset
  const int cur = p.cur_from_new ? w.hi - 1 : -1;

  for (int i = 0; i < my_n; ++i) {
    const int st = i % STAGES;
    if (!mbar_wait_bounded(bar0 + 8 * st, (i / STAGES) & 1)) {
      if (lane == 0) set_status(p.status, OL_DEVICE_GUARD);
      break;
    }
    const int t0 = w.t_begin + (warp + i * NWARPS) * kTok;
    uint8_t* sK = my_stages + st * kStageBytes;
    uint8_t* sV = sK + kPlaneBytes;

    if (cur >= t0 && cur < t0 + kTok) {
      // the token being appended: its K/V come from new_kv (the cache row is
      // stale); patch the tile and, for a fused step, store the row in the cache
      const int r = cur - t0;
      const int h = lane >> 4, c8 = (lane & 15) >> 1, sub = (lane & 1) * 8;
      const int off = h * kHalfBytes + r * 128 + ((c8 ^ (r & 7)) << 4) + sub;
      const uint2* nk = reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.new_kv) +
                                                       ((size_t)w.b * p.kv_heads + w.g) * 128) + lane;
      const uint2* nv = reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.new_kv) +
                                                       (((size_t)p.batch + w.b) * p.kv_heads + w.g) * 128) + lane;
      const uint2 kv = *nk, vv = *nv;
      *reinterpret_cast<uint2*>(sK + off) = kv;
      *reinterpret_cast<uint2*>(sV + off) = vv;
      if (p.append) {
        uint16_t* base = reinterpret_cast<uint16_t*>(PAGED ? p.pool : p.cache);
        bool bad = false;
        const int rowk = tile_row(p, PAGED, 0, w.b, w.g, t0, &bad) + r;
        const int rowv = tile_row(p, PAGED, 1, w.b, w.g, t0, &bad) + r;
        if (!bad) {
          reinterpret_cast<uint2*>(base + (size_t)rowk * 128)[lane] = kv;
          reinterpret_cast<uint2*>(base + (size_t)rowv * 128)[lane] = vv;
        }
      }
    }
    const int rv_hi = w.hi - t0;  // V rows >= rv_hi are outside the valid range: zero them
    if (rv_hi < kTok) {
      for (int idx = lane; idx < (kTok - rv_hi) * 16; idx += 32) {
        const int r = rv_hi + (idx >> 4), cc = idx & 15;
        *reinterpret_cast<uint4*>(sV + (cc >> 3) * kHalfBytes + r * 128 + (cc & 7) * 16) = make_uint4(0, 0, 0, 0);
      }
    }
    __syncwarp();

    // S^T = K q^T
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t kbase = smem_u32(sK);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int ch = 2 * kk + cK;
      uint32_t a0, a1, a2, a3;
      ldsm_x4(kbase + (ch >> 3) * kHalfBytes + rK * 128 + (((ch & 7) ^ r8) << 4), a0, a1, a2, a3);
      mma_bf16_16816(s, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
    }
    // s[0]: (token n, head 2c)  s[1]: (token n, head 2c+1)  s[2], s[3]: token n + 8
    const int ta = t0 + n, tb = ta + 8;
    const bool va = ta >= w.lo && ta < w.t_end, vb = tb >= w.lo && tb < w.t_end;
    const float s00 = va ? s[0] * p.scale_log2 : -INFINITY;
    const float s01 = va ? s[1] * p.scale_log2 : -INFINITY;
    const float s10 = vb ? s[2] * p.scale_log2 : -INFINITY;
    const float s11 = vb ? s[3] * p.scale_log2 : -INFINITY;
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
    // P^T as the B operand (16 tokens x 8 heads), carried as bf16 hi + bf16 lo
    // (p - hi) so the P.V product keeps ~16 significant bits of each weight
    const uint32_t h0 = pack_bf16x2(p00, p01), h1 = pack_bf16x2(p10, p11);
    const uint32_t l0 = pack_bf16x2(p00 - __uint_as_float(h0 << 16), p01 - __uint_as_float(h0 & 0xffff0000u));
    const uint32_t l1 = pack_bf16x2(p10 - __uint_as_float(h1 << 16), p11 - __uint_as_float(h1 & 0xffff0000u));
    const uint32_t ph0 = movmatrix_trans(h0), ph1 = movmatrix_trans(h1);
    const uint32_t pl0 = movmatrix_trans(l0), pl1 = movmatrix_trans(l1);
    const uint32_t vbase = smem_u32(sV);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int ch = 2 * mt + cV;
      uint32_t a0, a1, a2, a3;
      ldsm_x4_trans(vbase + (ch >> 3) * kHalfBytes + rV * 128 + (((ch & 7) ^ r8) << 4), a0, a1, a2, a3);
      mma_bf16_16816(o[mt], a0, a1, a2, a3, ph0, ph1);
      mma_bf16_16816(o[mt], a0, a1, a2, a3, pl0, pl1);
    }
    __syncwarp();
    if (lane == 0 && i + STAGES < my_n) {
      fence_proxy_async_smem();  // generic writes to this stage (patch, zeroing) before the async-proxy refill
      issue(i + STAGES);
    }
  }

  // per-warp state into the warp's own first stage, then the CTA / cluster / split merge
  store_warp_state(reinterpret_cast<float*>(my_stages), ms, warp, o, m_run0, m_run1, l_run0, l_run1);
  float* merged = reinterpret_cast<float*>(stages + kStageBytes);  // warp 0's second stage (no cluster)
  merge_and_finish(
      p, w, NWARPS,
      [&](int st) { return reinterpret_cast<const float*>(stages + st * STAGES * kStageBytes); }, merged,
      cmerged, ms);
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

// 2D view of a bf16 buffer as rows of 128 elements; boxes of 16 rows x 64 elements, 128B swizzle.
bool encode_rows128(CUtensorMap* map, void* base, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, rows};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, kTok};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NWARPS, int STAGES, bool PAGED>
cudaError_t ensure_attrs() {
  static cudaError_t state = [] {
    auto kern = fast_bf16_kernel<NWARPS, STAGES, PAGED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FastLayout<NWARPS, STAGES>::kTotal);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
  }();
  return state;
}

// Largest cluster size in {16, 8, 4, 2, 1} that the device can co-schedule for this kernel.
template <int NWARPS, int STAGES, bool PAGED>
int max_cluster() {
  static int cs = [] {
    if (ensure_attrs<NWARPS, STAGES, PAGED>() != cudaSuccess) return 1;
    for (int c = 16; c >= 2; c >>= 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(c, 1, 1);
      cfg.blockDim = dim3(NWARPS * 32, 1, 1);
      cfg.dynamicSmemBytes = FastLayout<NWARPS, STAGES>::kTotal;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = c;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, fast_bf16_kernel<NWARPS, STAGES, PAGED>, &cfg) == cudaSuccess && n > 0)
        return c;
      cudaGetLastError();
    }
    return 1;
  }();
  return cs;
}

template <int NWARPS, int STAGES, bool PAGED>
cudaError_t launch_cfg(const CUtensorMap& map, const AttnParams& p, cudaStream_t s) {
  auto kern = fast_bf16_kernel<NWARPS, STAGES, PAGED>;
  constexpr int smem = FastLayout<NWARPS, STAGES>::kTotal;
  cudaError_t e = ensure_attrs<NWARPS, STAGES, PAGED>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  const bool chunk = p.nq > 1;  // query tokens along x, the plan's CTAs (and clusters) along y
  cfg.gridDim = chunk ? dim3(p.nq, p.total_ctas, 1) : dim3(p.total_ctas, 1, 1);
  cfg.blockDim = dim3(NWARPS * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = chunk ? 1 : p.cluster;
  attr[1].val.clusterDim.y = chunk ? p.cluster : 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, map, p);
}

template <bool PAGED>
cudaError_t launch_variant(const CUtensorMap& map, const AttnParams& p, cudaStream_t s) {
  switch (p.variant) {
    case 1: return launch_cfg<4, 3, PAGED>(map, p, s);
    case 2: return launch_cfg<4, 2, PAGED>(map, p, s);
    case 3: return launch_cfg<8, 2, PAGED>(map, p, s);
    default: return launch_cfg<4, 4, PAGED>(map, p, s);
  }
}

}  // namespace

int fast_bf16_smem(int variant) {
  switch (variant) {
    case 1: return FastLayout<4, 3>::kTotal;
    case 2: return FastLayout<4, 2>::kTotal;
    case 3: return FastLayout<8, 2>::kTotal;
    default: return FastLayout<4, 4>::kTotal;
  }
}

int fast_bf16_warps(int variant) { return variant == 3 ? 8 : 4; }

int fast_bf16_max_cluster(int variant, bool paged) {
  switch (variant) {
    case 1: return paged ? max_cluster<4, 3, true>() : max_cluster<4, 3, false>();
    case 2: return paged ? max_cluster<4, 2, true>() : max_cluster<4, 2, false>();
    case 3: return paged ? max_cluster<8, 2, true>() : max_cluster<8, 2, false>();
    default: return paged ? max_cluster<4, 4, true>() : max_cluster<4, 4, false>();
  }
}

bool fast_bf16_supported(const AttnParams& p) {
  if (p.dtype != OL_BF16 || p.head_dim != 128 || p.group > 8) return false;
  // TMA row coordinates are 32-bit
  const unsigned long long rows = p.layout == OL_LAYOUT_PAGED ? 2ull * p.num_pages * p.kv_heads * p.page_size
                                                              : 2ull * p.batch * p.kv_heads * p.capacity;
  if (rows >= (1ull << 31)) return false;
  if (p.layout == OL_LAYOUT_CONTIGUOUS) return true;
  if (p.layout == OL_LAYOUT_PAGED) return p.page_size % kTok == 0;
  return false;
}

cudaError_t launch_fast_bf16(const AttnParams& p, cudaStream_t s) {
  if (p.total_ctas <= 0) return cudaSuccess;
  CUtensorMap map;
  const bool paged = p.layout == OL_LAYOUT_PAGED;
  const uint64_t rows = paged ? 2ull * p.num_pages * p.kv_heads * p.page_size
                              : 2ull * p.batch * p.kv_heads * p.capacity;
  if (!encode_rows128(&map, paged ? p.pool : p.cache, rows)) return cudaErrorInvalidValue;
  if (paged) return launch_variant<true>(map, p, s);
  return launch_variant<false>(map, p, s);
}

}  // namespace ol
