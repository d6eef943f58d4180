// ol_noalloc.cu -- ol_decode_step_noalloc: the fused decode step for callers
// that cannot allocate device memory. Its workspace is this file's static
// device array; nothing is allocated per call.
#include <mutex>

#include <cuda_runtime.h>

#include "ol_internal.h"
#include "ol_launch.h"

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

}  // namespace

extern "C" ol_status ol_decode_step_noalloc(int32_t layout, const void* cache_desc, void* updated, const void* q,
                                            int32_t q_heads, const void* new_kv, const int32_t* lens_host,
                                            const int32_t* lens_dev, float scale, int32_t window, void* out,
                                            int32_t out_dtype, ol_stream stream) {
  void* scratch = scratch_for_current_device();
  if (!scratch) return OL_ERR_CUDA;
  // Every check of ol_decode_step first (the scratch size included: a request
  // whose workspace exceeds it is OL_ERR_WORKSPACE), so a rejected call
  // enqueues nothing and returns what ol_decode_step would.
  ol_status st = ol::decode_step_impl(layout, cache_desc, updated, q, q_heads, new_kv, lens_host, lens_dev, scale,
                                      window, out, out_dtype, scratch, OL_NOALLOC_SCRATCH_BYTES, stream, true);
  if (st != OL_OK) return st;
  // The status word and the ticket counters must start at zero (an earlier
  // call may have been cut short); the partials are written before they are read.
  int32_t batch = 0, kv_heads = 0;
  switch (layout) {
    case OL_LAYOUT_CONTIGUOUS:
      batch = static_cast<const ol_kv_cache*>(cache_desc)->batch;
      kv_heads = static_cast<const ol_kv_cache*>(cache_desc)->kv_heads;
      break;
    case OL_LAYOUT_PAGED:
      batch = static_cast<const ol_paged_kv*>(cache_desc)->batch;
      kv_heads = static_cast<const ol_paged_kv*>(cache_desc)->kv_heads;
      break;
    case OL_LAYOUT_INT4:
      batch = static_cast<const ol_int4_kv*>(cache_desc)->batch;
      kv_heads = static_cast<const ol_int4_kv*>(cache_desc)->kv_heads;
      break;
    default:  // not reached: the checks above accept only the three layouts
      return OL_ERR_UNSUPPORTED;
  }
  const size_t zero_bytes = ol::partials_offset(batch, kv_heads);
  if (cudaMemsetAsync(scratch, 0, zero_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess) return OL_ERR_CUDA;
  return ol_decode_step(layout, cache_desc, updated, q, q_heads, new_kv, lens_host, lens_dev, scale, window, out,
                        out_dtype, scratch, OL_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" ol_status ol_noalloc_status(int32_t* status_out, ol_stream stream) {
  if (!status_out) return OL_ERR_NULL;
  void* scratch = scratch_for_current_device();
  if (!scratch) return OL_ERR_CUDA;
  return ol_workspace_status(scratch, status_out, stream);
}
