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
#if defined(OL_PHASE_STAMPS) && OL_PHASE_STAMPS
// Timing build: thread 0 of every decode-kernel CTA records (%globaltimer,
// clock64) at each phase boundary into a ring of 64 launches x 256 CTAs. The
// launch index is a running CTA count divided by the grid size: every CTA of a
// launch starts (and counts itself) before any CTA of the next launch, which
// programmatic dependent launch starts only once all of them have triggered.
namespace ol {
enum { OL_PH_ENTRY, OL_PH_WAIT, OL_PH_INPUTS, OL_PH_FIRST_TILE, OL_PH_TILES, OL_PH_ALL_TILES, OL_PH_CTA_MERGED,
       OL_PH_CLUSTER, OL_PH_END, OL_PH_COUNT };
constexpr int kStampSteps = 64, kStampCtas = 256;
__device__ unsigned long long g_stamps[kStampSteps][kStampCtas][OL_PH_COUNT][2];
__device__ unsigned int g_stamp_seq;
__shared__ unsigned int s_stamp_slot;
__device__ __forceinline__ void stamp_record(int ph) {
  const unsigned slot = s_stamp_slot;
  if (slot == 0xffffffffu) return;
  unsigned long long t, c;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
  g_stamps[slot / kStampCtas][slot % kStampCtas][ph][0] = t;
  g_stamps[slot / kStampCtas][slot % kStampCtas][ph][1] = c;
}
__device__ __forceinline__ void stamp_begin(bool on) {
  if (threadIdx.x != 0) return;
  unsigned slot = 0xffffffffu;
  if (on && blockIdx.x < (unsigned)kStampCtas) {
    const unsigned seq = atomicAdd(&g_stamp_seq, 1u);
    slot = (seq / (gridDim.x * gridDim.y * gridDim.z)) % kStampSteps * kStampCtas + blockIdx.x;
  }
  s_stamp_slot = slot;
  stamp_record(OL_PH_ENTRY);
}
}  // namespace ol
#define OL_STAMP(ph) \
  do {               \
    if (threadIdx.x == 0) ::ol::stamp_record(::ol::ph); \
  } while (0)
// the stamp waits for `reg` (a loaded value) to arrive
#define OL_STAMP_AFTER(ph, reg)                                  \
  do {                                                           \
    if (threadIdx.x == 0) {                                      \
      uint32_t dep_;                                             \
      asm volatile("mov.b32 %0, %1;" : "=r"(dep_) : "r"(reg));   \
      ::ol::stamp_record(::ol::ph);                              \
    }                                                            \
  } while (0)
#define OL_STAMP_BEGIN(on) ::ol::stamp_begin(on)
#define OL_STAMP_END()  \
  do {                  \
    __syncthreads();    \
    OL_STAMP(OL_PH_END); \
  } while (0)
#endif

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

#define OL_CHUNK 0
constexpr float kLazy = 8.f;  // log2 headroom of the lazy softmax maximum

#define OL_FAST_KERNEL fast_bf16_kernel
#include "ol_fast_bf16_kernel.inc"
#undef OL_FAST_KERNEL
#undef OL_CHUNK
#define OL_CHUNK 1
#define OL_FAST_KERNEL fast_bf16_chunk_kernel
#include "ol_fast_bf16_kernel.inc"
#undef OL_FAST_KERNEL
#undef OL_CHUNK

// the decode or the chunked-step kernel of a variant
template <int NWARPS, int STAGES, bool PAGED, bool CHUNK>
constexpr auto kernel_of() {
  if constexpr (CHUNK)
    return fast_bf16_chunk_kernel<NWARPS, STAGES, PAGED>;
  else
    return fast_bf16_kernel<NWARPS, STAGES, PAGED>;
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

template <int NWARPS, int STAGES, bool PAGED, bool CHUNK = false>
cudaError_t ensure_attrs() {
  static cudaError_t state = [] {
    auto kern = kernel_of<NWARPS, STAGES, PAGED, CHUNK>();
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

// Clusters of cs CTAs of this kernel the device holds at once (0 if none).
template <int NWARPS, int STAGES, bool PAGED>
int active_clusters(int cs) {
  static int cached[17] = {0};
  static bool done[17] = {false};
  if (cs < 1 || cs > 16) return 0;
  if (!done[cs]) {
    int n = 0;
    if (ensure_attrs<NWARPS, STAGES, PAGED>() == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(cs, 1, 1);
      cfg.blockDim = dim3(NWARPS * 32, 1, 1);
      cfg.dynamicSmemBytes = FastLayout<NWARPS, STAGES>::kTotal;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cs;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, fast_bf16_kernel<NWARPS, STAGES, PAGED>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
    }
    cached[cs] = n;
    done[cs] = true;
  }
  return cached[cs];
}

template <int NWARPS, int STAGES, bool PAGED, bool CHUNK>
cudaError_t launch_cfg(const CUtensorMap& map, const AttnParams& p, cudaStream_t s) {
  auto kern = kernel_of<NWARPS, STAGES, PAGED, CHUNK>();
  constexpr int smem = FastLayout<NWARPS, STAGES>::kTotal;
  cudaError_t e = ensure_attrs<NWARPS, STAGES, PAGED, CHUNK>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  constexpr bool chunk = CHUNK;  // query-token slices along x, the plan's CTAs (and clusters) along y
  const int slices = chunk ? (p.nq + (p.tq > 1 ? p.tq : 1) - 1) / (p.tq > 1 ? p.tq : 1) : 1;
  cfg.gridDim = chunk ? dim3((slices + 1) / 2, p.total_ctas, 1) : dim3(p.total_ctas, 1, 1);  // 2 slices per CTA
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
  if (p.nq > 1)  // chunked steps: the two default variants (the plan keeps to them)
    return p.variant == 2 ? launch_cfg<4, 2, PAGED, true>(map, p, s) : launch_cfg<8, 2, PAGED, true>(map, p, s);
  switch (p.variant) {
    case 1: return launch_cfg<4, 3, PAGED, false>(map, p, s);
    case 2: return launch_cfg<4, 2, PAGED, false>(map, p, s);
    case 3: return launch_cfg<8, 2, PAGED, false>(map, p, s);
    case 4: return launch_cfg<6, 2, PAGED, false>(map, p, s);
    default: return launch_cfg<4, 4, PAGED, false>(map, p, s);
  }
}

}  // namespace

int fast_bf16_smem(int variant) {
  switch (variant) {
    case 1: return FastLayout<4, 3>::kTotal;
    case 2: return FastLayout<4, 2>::kTotal;
    case 3: return FastLayout<8, 2>::kTotal;
    case 4: return FastLayout<6, 2>::kTotal;
    default: return FastLayout<4, 4>::kTotal;
  }
}

int fast_bf16_warps(int variant) { return variant == 3 ? 8 : variant == 4 ? 6 : 4; }

int fast_bf16_max_cluster(int variant, bool paged) {
  switch (variant) {
    case 1: return paged ? max_cluster<4, 3, true>() : max_cluster<4, 3, false>();
    case 2: return paged ? max_cluster<4, 2, true>() : max_cluster<4, 2, false>();
    case 3: return paged ? max_cluster<8, 2, true>() : max_cluster<8, 2, false>();
    case 4: return paged ? max_cluster<6, 2, true>() : max_cluster<6, 2, false>();
    default: return paged ? max_cluster<4, 4, true>() : max_cluster<4, 4, false>();
  }
}

int fast_bf16_active_clusters(int variant, bool paged, int cs) {
  switch (variant) {
    case 1: return paged ? active_clusters<4, 3, true>(cs) : active_clusters<4, 3, false>(cs);
    case 2: return paged ? active_clusters<4, 2, true>(cs) : active_clusters<4, 2, false>(cs);
    case 3: return paged ? active_clusters<8, 2, true>(cs) : active_clusters<8, 2, false>(cs);
    case 4: return paged ? active_clusters<6, 2, true>(cs) : active_clusters<6, 2, false>(cs);
    default: return paged ? active_clusters<4, 4, true>(cs) : active_clusters<4, 4, false>(cs);
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

#if defined(OL_PHASE_STAMPS) && OL_PHASE_STAMPS
// Copy the timing build's stamp ring to host memory ([64][256][9][2] uint64:
// launch slot, CTA, phase, {%globaltimer ns, clock64}); with reset != 0 then
// zero it and restart the launch count (synchronizes the device).
extern "C" OL_API ol_status ol_debug_phase_stamps(void* host_out, size_t bytes, int32_t reset) {
  if (host_out && bytes > 0) {
    if (bytes > sizeof(ol::g_stamps)) bytes = sizeof(ol::g_stamps);
    if (cudaMemcpyFromSymbol(host_out, ol::g_stamps, bytes) != cudaSuccess) return OL_ERR_CUDA;
  }
  if (reset) {
    static unsigned long long zeros[ol::kStampCtas * ol::OL_PH_COUNT * 2];
    for (int s = 0; s < ol::kStampSteps; ++s)
      if (cudaMemcpyToSymbol(ol::g_stamps, zeros, sizeof(zeros), (size_t)s * sizeof(zeros)) != cudaSuccess)
        return OL_ERR_CUDA;
    const unsigned int z = 0;
    if (cudaMemcpyToSymbol(ol::g_stamp_seq, &z, sizeof(z)) != cudaSuccess) return OL_ERR_CUDA;
  }
  return cudaDeviceSynchronize() == cudaSuccess ? OL_OK : OL_ERR_CUDA;
}
#endif
