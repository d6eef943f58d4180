// ol_hpaged.cu -- the heterogeneous paged cache's append and selected-page
// conversion. Attention over it runs in the CUDA-core kernel (ol_generic.cu),
// which decodes every page with its own formats.
#include "ol_hpaged.cuh"

namespace ol {
namespace {

// One warp per (row, head, new token, plane): encode the token into its page.
// A page whose first slot lies inside this append is started by it and takes
// p.new_fmt (the token in slot 0 records that in the page's descriptor);
// other pages keep their formats. Positions or pages outside the cache (which
// the host rejects) are skipped on the device.
__global__ void hpaged_append_kernel(const AppendParams p) {
  const int j = blockIdx.x % p.new_len;
  const int h = (blockIdx.x / p.new_len) % p.kv_heads;
  const int b = blockIdx.x / (p.new_len * p.kv_heads);
  const int plane = blockIdx.y;
  const int S = p.page_size, D = p.head_dim;
  int pos = p.positions[b];
  if (p.positions_are_lens) pos -= p.new_len;
  const int t = pos + j;
  if (pos < 0 || t >= p.max_pages * S) return;  // device guard
  const int page = p.block_table[(size_t)b * p.max_pages + t / S];
  if (page < 0 || page >= p.num_pages) return;  // device guard
  const int s = t % S;
  const bool started = t - s >= pos;  // the page's slot 0 is part of this append
  const ol_plane_format pf = started ? (plane == 0 ? p.new_fmt.k : p.new_fmt.v)
                                     : (plane == 0 ? p.page_fmt[page].k : p.page_fmt[page].v);
  const uint16_t* x = reinterpret_cast<const uint16_t*>(p.values) +
                      ((((size_t)plane * p.batch + b) * p.kv_heads + h) * p.new_len + j) * D;
  uint8_t* row = hp_row(reinterpret_cast<uint8_t*>(p.pool), p.kv_heads, S, D, page, plane, h, s, pf.format);
  hp_encode_row_warp([&](int d) { return bf16_bits_to_float(x[d]); }, D, pf, row);
  if (s == 0 && h == 0 && (threadIdx.x & 31) == 0) {
    if (plane == 0)
      p.page_fmt[page].k = pf;
    else
      p.page_fmt[page].v = pf;
  }
}

// One CTA per (selected page, plane). A head's rows are decoded into shared
// memory before any of them is rewritten, and the heads are taken in the order
// in which no head's new rows cover another head's unread rows: from the last
// head down when the target rows are wider, from the first up otherwise.
__global__ void hpaged_quantize_kernel(const QuantizeParams p) {
  extern __shared__ float vals[];  // [page_size][head_dim]
  const int i = blockIdx.x, plane = blockIdx.y;
  const int page = p.pages[i];
  const int S = p.page_size, D = p.head_dim, H = p.kv_heads;
  if (page < 0 || page >= p.num_pages) return;  // device guard (the host checked the same indices)
  const int nvalid = min(max(p.valid[i], 0), S);
  const ol_plane_format from = plane == 0 ? p.page_fmt[page].k : p.page_fmt[page].v;
  const ol_plane_format to = plane == 0 ? p.to.k : p.to.v;
  const bool wider = fmt_row_bytes(to.format, D) > fmt_row_bytes(from.format, D);
  uint8_t* pool = p.pool;
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int k = 0; k < H; ++k) {
    const int h = wider ? H - 1 - k : k;
    for (int e = threadIdx.x; e < S * D; e += blockDim.x) {
      const int s = e / D, d = e % D;
      vals[e] = s < nvalid ? hp_decode(hp_row(pool, H, S, D, page, plane, h, s, from.format), d, from) : 0.f;
    }
    __syncthreads();
    for (int s = warp; s < S; s += nwarps)
      hp_encode_row_warp([&](int d) { return vals[s * D + d]; }, D, to,
                         hp_row(pool, H, S, D, page, plane, h, s, to.format));
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (plane == 0)
      p.page_fmt[page].k = to;
    else
      p.page_fmt[page].v = to;
  }
}

}  // namespace

cudaError_t launch_hpaged_append(const AppendParams& p, cudaStream_t s) {
  if (p.batch == 0 || p.new_len == 0) return cudaSuccess;
  dim3 grid(p.batch * p.kv_heads * p.new_len, 2);
  hpaged_append_kernel<<<grid, 32, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_hpaged_quantize(const QuantizeParams& p, cudaStream_t s) {
  if (p.n == 0) return cudaSuccess;
  const size_t smem = (size_t)p.page_size * p.head_dim * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(hpaged_quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  hpaged_quantize_kernel<<<dim3(p.n, 2), 256, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ol
