// ol_noalloc.cu -- ol_decode_step_noalloc: the fused decode step for callers
// that cannot allocate device memory. Its workspace is this file's static
// device array; nothing is allocated per call.
#include <mutex>

#include <cuda_runtime.h>

#include "ol_internal.h"

namespace {

// Shared scratch of every ol_decode_step_noalloc call in this process (per device).
static __device__ __align__(256) unsigned char g_noalloc_scratch[OL_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current). Returns nullptr on failure.
void* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

ol_status sizes_of(int32_t layout, const void* desc, int32_t* batch, int32_t* kv_heads, int32_t* head_dim) {
  if (!desc) return OL_ERR_NULL;
  switch (layout) {
    case OL_LAYOUT_CONTIGUOUS: {
      const ol_kv_cache* c = static_cast<const ol_kv_cache*>(desc);
      *batch = c->batch, *kv_heads = c->kv_heads, *head_dim = c->head_dim;
      return OL_OK;
    }
    case OL_LAYOUT_PAGED: {
      const ol_paged_kv* c = static_cast<const ol_paged_kv*>(desc);
      *batch = c->batch, *kv_heads = c->kv_heads, *head_dim = c->head_dim;
      return OL_OK;
    }
    case OL_LAYOUT_INT4: {
      const ol_int4_kv* c = static_cast<const ol_int4_kv*>(desc);
      *batch = c->batch, *kv_heads = c->kv_heads, *head_dim = c->head_dim;
      return OL_OK;
    }
    default:
      return OL_ERR_UNSUPPORTED;
  }
}

}  // namespace

extern "C" ol_status ol_decode_step_noalloc(int32_t layout, const void* cache_desc, void* updated, const void* q,
                                            int32_t q_heads, const void* new_kv, const int32_t* lens_host,
                                            const int32_t* lens_dev, float scale, int32_t window, void* out,
                                            int32_t out_dtype, ol_stream stream) {
  int32_t batch = 0, kv_heads = 0, head_dim = 0;
  ol_status st = sizes_of(layout, cache_desc, &batch, &kv_heads, &head_dim);
  if (st != OL_OK) return st;
  if (batch < 0 || kv_heads <= 0 || head_dim <= 0 || q_heads <= 0 || q_heads % kv_heads != 0) return OL_ERR_SHAPE;
  const size_t need = ol::workspace_bytes(batch, q_heads, kv_heads, head_dim);
  if (need > OL_NOALLOC_SCRATCH_BYTES) return OL_ERR_WORKSPACE;
  void* scratch = scratch_for_current_device();
  if (!scratch) return OL_ERR_CUDA;
  // The ticket counters and status word must start at zero; the partials are
  // always written before they are read.
  const size_t zero_bytes = ol::partials_offset(batch, kv_heads);
  if (cudaMemsetAsync(scratch, 0, zero_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess) return OL_ERR_CUDA;
  return ol_decode_step(layout, cache_desc, updated, q, q_heads, new_kv, lens_host, lens_dev, scale, window, out,
                        out_dtype, scratch, OL_NOALLOC_SCRATCH_BYTES, stream);
}
