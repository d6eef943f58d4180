// ol_append.cu -- the in-place appends on their own: CacheUpdate on a
// contiguous cache, PagedCacheUpdate through a block table, and the INT4
// quantize-and-append. Each writes only the rows [p_b, p_b + new_len) of its
// rows; positions that disagree with the host-validated bounds are skipped on
// the device, never written out of bounds.
#include "ol_common.cuh"

namespace ol {
namespace {

// One CTA per (plane, row, head, new token): copy one D-element row.
template <typename T>
__global__ void copy_rows_kernel(const AppendParams p) {
  const int j = blockIdx.x % p.new_len;
  const int h = (blockIdx.x / p.new_len) % p.kv_heads;
  const int b = blockIdx.x / (p.new_len * p.kv_heads);
  const int plane = blockIdx.y;
  const int D = p.head_dim;
  int pos = p.positions ? p.positions[b] : p.scalar_position;
  if (p.positions_are_lens) pos -= p.new_len;
  if (pos < 0 || (long long)pos + p.new_len > p.capacity) return;  // device guard
  const int t = pos + j;
  size_t dst;
  T* base;
  if (p.layout == OL_LAYOUT_CONTIGUOUS) {
    base = reinterpret_cast<T*>(p.cache);
    dst = ((((size_t)plane * p.batch + b) * p.kv_heads + h) * p.capacity + t) * D;
  } else {
    int page = p.block_table[(size_t)b * p.max_pages + t / p.page_size];
    if (page < 0 || page >= p.num_pages) return;  // device guard
    base = reinterpret_cast<T*>(p.pool);
    dst = ((((size_t)plane * p.num_pages + page) * p.kv_heads + h) * p.page_size + t % p.page_size) * D;
  }
  const size_t src = ((((size_t)plane * p.batch + b) * p.kv_heads + h) * p.new_len + j) * D;
  const T* in = reinterpret_cast<const T*>(p.values);
  for (int d = threadIdx.x; d < D; d += blockDim.x) base[dst + d] = in[src + d];
}

// One warp per (plane, row, head, new token): quantize the token and store its INT4 row.
__global__ void int4_append_kernel(const AppendParams p) {
  const int j = blockIdx.x % p.new_len;
  const int h = (blockIdx.x / p.new_len) % p.kv_heads;
  const int b = blockIdx.x / (p.new_len * p.kv_heads);
  const int plane = blockIdx.y;
  const int D = p.head_dim;
  int pos = p.positions[b];
  if (p.positions_are_lens) pos -= p.new_len;
  if (pos < 0 || (long long)pos + p.new_len > p.capacity) return;  // device guard
  const size_t row = (((size_t)plane * p.batch + b) * p.kv_heads + h) * p.capacity + pos + j;
  const size_t src = ((((size_t)plane * p.batch + b) * p.kv_heads + h) * p.new_len + j) * D;
  int4_quantize_row_warp(reinterpret_cast<const uint16_t*>(p.values) + src, D, p.quant_mode, p.fixed_scale,
                         p.fixed_zp, p.codes + row * (D / 2), p.scales + row * (D / 32),
                         p.zps + row * (D / 64));
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t s) {
  if (p.batch == 0 || p.new_len == 0) return cudaSuccess;
  if (p.layout == OL_LAYOUT_INT4) {
    dim3 grid(p.batch * p.kv_heads * p.new_len, 2);
    int4_append_kernel<<<grid, 32, 0, s>>>(p);
    return cudaGetLastError();
  }
  dim3 grid(p.batch * p.kv_heads * p.new_len, 2);
  int threads = p.head_dim >= 128 ? 128 : 32;
  if (p.dtype == OL_F32)
    copy_rows_kernel<float><<<grid, threads, 0, s>>>(p);
  else
    copy_rows_kernel<uint16_t><<<grid, threads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ol
