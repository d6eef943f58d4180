// ol_generic.cu -- CUDA-core decode attention for every layout and dtype:
// contiguous fp32/bf16, paged fp32/bf16, INT4 and heterogeneous pages (each
// page decoded by its own formats), any head_dim up to 256, any GQA group. It serves the shapes the tensor-core kernels do not take (for
// example fp32 caches with head_dim 4) with the same split plan, merge and
// fused append as they use.
//
// One CTA = (row b, kv head g, split s, block of up to 4 query heads). Each
// warp walks tokens t = t_begin + warp, + 4, ...; every lane owns head_dim/32
// dimensions; per token the warp reduces q.k with shuffles and updates an
// online-softmax state (m, l, o) per query head. Warps merge in shared memory
// and the CTA finishes through the split-K ticket (finish_split).
#include <climits>

#include "ol_hpaged.cuh"

namespace ol {
namespace {

constexpr int kGenWarps = 4;
constexpr int kGenHeads = 4;
constexpr int kMaxDpl = 8;  // dims per lane: head_dim <= 256

// Element d of token t of kv head g of row b, plane 0 (K) or 1 (V), as fp32.
__device__ __forceinline__ float load_kv(const AttnParams& p, int plane, int b, int g, int t, int d) {
  const int D = p.head_dim;
  if (p.layout == OL_LAYOUT_CONTIGUOUS) {
    size_t idx = ((((size_t)plane * p.batch + b) * p.kv_heads + g) * p.capacity + t) * D + d;
    return p.dtype == OL_F32 ? reinterpret_cast<const float*>(p.cache)[idx]
                             : bf16_bits_to_float(reinterpret_cast<const uint16_t*>(p.cache)[idx]);
  }
  if (p.layout == OL_LAYOUT_PAGED) {
    int page = p.block_table[(size_t)b * p.max_pages + t / p.page_size];
    if (page < 0 || page >= p.num_pages) {  // device guard: never read outside the pool
      set_status(p.status, OL_DEVICE_GUARD);
      return 0.f;
    }
    size_t idx = ((((size_t)plane * p.num_pages + page) * p.kv_heads + g) * p.page_size +
                  t % p.page_size) * D + d;
    return p.dtype == OL_F32 ? reinterpret_cast<const float*>(p.pool)[idx]
                             : bf16_bits_to_float(reinterpret_cast<const uint16_t*>(p.pool)[idx]);
  }
  if (p.layout == OL_LAYOUT_HPAGED) {
    int page = p.block_table[(size_t)b * p.max_pages + t / p.page_size];
    if (page < 0 || page >= p.num_pages) {
      set_status(p.status, OL_DEVICE_GUARD);
      return 0.f;
    }
    const ol_plane_format pf = plane == 0 ? p.page_fmt[page].k : p.page_fmt[page].v;
    return hp_decode(hp_row(reinterpret_cast<uint8_t*>(p.pool), p.kv_heads, p.page_size, D, page, plane, g,
                            t % p.page_size, pf.format),
                     d, pf);
  }
  // INT4: (code - zp) * scale
  size_t row = (((size_t)plane * p.batch + b) * p.kv_heads + g) * p.capacity + t;
  uint8_t cb = p.codes[row * (D / 2) + d / 2];
  int code = (d & 1) ? (cb >> 4) : (cb & 0xF);
  int blk = d / 32;
  uint8_t zb = p.zps[row * (D / 64) + blk / 2];
  int zp = (blk & 1) ? (zb >> 4) : (zb & 0xF);
  float s = fp16_bits_to_float(p.scales[row * (D / 32) + blk]);
  return static_cast<float>(code - zp) * s;
}

// New token j of row b (the one a fused step appends, or token j of a chunk
// whose tokens are attended uncompressed), from new_kv [2, B, Hkv, nq, D].
__device__ __forceinline__ float load_new(const AttnParams& p, int plane, int b, int g, int j, int d) {
  size_t idx = ((((size_t)plane * p.batch + b) * p.kv_heads + g) * (p.nq > 1 ? p.nq : 1) + j) * p.head_dim + d;
  if (p.dtype == OL_F32 && p.layout != OL_LAYOUT_INT4) return reinterpret_cast<const float*>(p.new_kv)[idx];
  return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(p.new_kv)[idx]);
}

// Write the appended token of (b, g) at position pos into the cache (one warp).
__device__ void append_token_warp(const AttnParams& p, int b, int g, int pos) {
  const int lane = threadIdx.x & 31;
  const int D = p.head_dim;
  for (int plane = 0; plane < 2; ++plane) {
    size_t src = (((size_t)plane * p.batch + b) * p.kv_heads + g) * D;
    if (p.layout == OL_LAYOUT_INT4) {
      size_t row = (((size_t)plane * p.batch + b) * p.kv_heads + g) * p.capacity + pos;
      int4_quantize_row_warp(reinterpret_cast<const uint16_t*>(p.new_kv) + src, D, p.quant_mode,
                             p.fixed_scale, p.fixed_zp, p.codes + row * (D / 2),
                             p.scales + row * (D / 32), p.zps + row * (D / 64));
      continue;
    }
    if (p.layout == OL_LAYOUT_HPAGED) {
      int page = p.block_table[(size_t)b * p.max_pages + pos / p.page_size];
      if (page < 0 || page >= p.num_pages) {
        if (lane == 0) set_status(p.status, OL_DEVICE_GUARD);
        return;
      }
      const int slot = pos % p.page_size;
      // a token in slot 0 starts its page, which takes the step's formats
      const ol_plane_format pf = slot == 0 ? (plane == 0 ? p.new_fmt.k : p.new_fmt.v)
                                           : (plane == 0 ? p.page_fmt[page].k : p.page_fmt[page].v);
      const uint16_t* x = reinterpret_cast<const uint16_t*>(p.new_kv) + src;
      hp_encode_row_warp([&](int d) { return bf16_bits_to_float(x[d]); }, D, pf,
                         hp_row(reinterpret_cast<uint8_t*>(p.pool), p.kv_heads, p.page_size, D, page, plane, g,
                                slot, pf.format));
      if (slot == 0 && g == 0 && lane == 0) {
        if (plane == 0)
          p.page_fmt[page].k = pf;
        else
          p.page_fmt[page].v = pf;
      }
      continue;
    }
    size_t dst;
    if (p.layout == OL_LAYOUT_CONTIGUOUS) {
      dst = ((((size_t)plane * p.batch + b) * p.kv_heads + g) * p.capacity + pos) * D;
    } else {
      int page = p.block_table[(size_t)b * p.max_pages + pos / p.page_size];
      if (page < 0 || page >= p.num_pages) {
        if (lane == 0) set_status(p.status, OL_DEVICE_GUARD);
        return;
      }
      dst = ((((size_t)plane * p.num_pages + page) * p.kv_heads + g) * p.page_size + pos % p.page_size) * D;
    }
    void* base = p.layout == OL_LAYOUT_CONTIGUOUS ? p.cache : p.pool;
    if (p.dtype == OL_F32) {
      for (int d = lane; d < D; d += 32)
        reinterpret_cast<float*>(base)[dst + d] = reinterpret_cast<const float*>(p.new_kv)[src + d];
    } else {
      for (int d = lane; d < D; d += 32)
        reinterpret_cast<uint16_t*>(base)[dst + d] = reinterpret_cast<const uint16_t*>(p.new_kv)[src + d];
    }
  }
}

__global__ void __launch_bounds__(kGenWarps * 32) generic_attn_kernel(const __grid_constant__ AttnParams p) {
  __shared__ Work sw;
  __shared__ int sm_flag, sm_new_lo;
  __shared__ float sm_wm[kGenWarps][kGenHeads], sm_wl[kGenWarps][kGenHeads];
  __shared__ float sm_wo[kGenWarps][kGenHeads][256];
  __shared__ float sm_m[kGenHeads], sm_l[kGenHeads];
  __shared__ float sm_o[kGenHeads][256];
  __shared__ float sm_scratch[2 * 256];

  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    Work w = p.inline_lens ? map_cta_warp(p.lens_inline, p.batch, p.kv_heads, p.capacity, p.window, p.chunk,
                                          cta_index(p), nullptr, 1, p.ordered ? p.row_order : nullptr)
                           : map_cta_warp(p.lens, p.batch, p.kv_heads, p.capacity, p.window, p.chunk, cta_index(p),
                                          p.status);
    const int row_hi = w.hi;  // the row's length: its new tokens are the last max(nq, 1)
    slice_query(w, p);
    if (lane == 0) {
      sw = w;
      sm_new_lo = row_hi - (p.nq > 1 ? p.nq : 1);
    }
  }
  __syncthreads();
  const Work w = sw;
  if (!w.valid) return;

  const int D = p.head_dim;
  const int G = p.group;
  const int heads_lo = head_block(p) * kGenHeads;
  const int heads_hi = min(G, heads_lo + kGenHeads);
  const int nh = heads_hi - heads_lo;
  // tokens from new_lo on come from new_kv when cur_from_new (the decode step's
  // current token, or every token of a chunk)
  const int new_lo = p.cur_from_new ? sm_new_lo : INT_MAX;

  float q[kGenHeads][kMaxDpl];
  float m[kGenHeads], l[kGenHeads], o[kGenHeads][kMaxDpl];
#pragma unroll
  for (int j = 0; j < kGenHeads; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxDpl; ++i) {
      o[j][i] = 0.f;
      int d = lane + 32 * i;
      float qv = 0.f;
      if (j < nh && d < D) {
        size_t qi = (((size_t)w.b * p.q_heads + (size_t)w.g * G + heads_lo + j) * (p.nq > 1 ? p.nq : 1) +
                     query_index(p)) * D + d;
        qv = (p.dtype == OL_F32 && p.layout != OL_LAYOUT_INT4)
                 ? reinterpret_cast<const float*>(p.q)[qi]
                 : bf16_bits_to_float(reinterpret_cast<const uint16_t*>(p.q)[qi]);
      }
      q[j][i] = qv;
    }
  }

  const int t_first = max(w.t_begin, w.lo);
  for (int t = t_first + warp; t < w.t_end; t += kGenWarps) {
    float k[kMaxDpl], v[kMaxDpl];
#pragma unroll
    for (int i = 0; i < kMaxDpl; ++i) {
      int d = lane + 32 * i;
      k[i] = 0.f;
      v[i] = 0.f;
      if (d < D) {
        if (t >= new_lo) {
          k[i] = load_new(p, 0, w.b, w.g, t - new_lo, d);
          v[i] = load_new(p, 1, w.b, w.g, t - new_lo, d);
        } else {
          k[i] = load_kv(p, 0, w.b, w.g, t, d);
          v[i] = load_kv(p, 1, w.b, w.g, t, d);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kGenHeads; ++j) {
      if (j >= nh) break;
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxDpl; ++i) s += q[j][i] * k[i];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      s *= p.scale_log2;
      float mn = fmaxf(m[j], s);
      float alpha = exp2f(m[j] - mn);
      float pw = exp2f(s - mn);
      l[j] = l[j] * alpha + pw;
#pragma unroll
      for (int i = 0; i < kMaxDpl; ++i) o[j][i] = o[j][i] * alpha + pw * v[i];
      m[j] = mn;
    }
  }

#pragma unroll
  for (int j = 0; j < kGenHeads; ++j) {
    if (lane == 0) {
      sm_wm[warp][j] = m[j];
      sm_wl[warp][j] = l[j];
    }
#pragma unroll
    for (int i = 0; i < kMaxDpl; ++i) {
      int d = lane + 32 * i;
      if (d < D) sm_wo[warp][j][d] = o[j][i];
    }
  }
  __syncthreads();
  if (threadIdx.x < nh) {
    int j = threadIdx.x;
    float M = -INFINITY;
    for (int ww = 0; ww < kGenWarps; ++ww) M = fmaxf(M, sm_wm[ww][j]);
    float L = 0.f;
    if (M != -INFINITY)
      for (int ww = 0; ww < kGenWarps; ++ww)
        if (sm_wm[ww][j] != -INFINITY) L += sm_wl[ww][j] * exp2f(sm_wm[ww][j] - M);
    sm_m[j] = M;
    sm_l[j] = L;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nh * D; i += blockDim.x) {
    int j = i / D, d = i % D;
    float M = sm_m[j], acc = 0.f;
    if (M != -INFINITY)
      for (int ww = 0; ww < kGenWarps; ++ww)
        if (sm_wm[ww][j] != -INFINITY) acc += sm_wo[ww][j][d] * exp2f(sm_wm[ww][j] - M);
    sm_o[j][d] = acc;
  }
  __syncthreads();

  // The fused append: the last split of (b, g) writes the new token. Nothing
  // in this launch reads that cache row (the attention takes it from new_kv).
  if (p.append && w.s == w.nsplit - 1 && head_block(p) == 0 && warp == 0 && w.hi >= 1)
    append_token_warp(p, w.b, w.g, w.hi - 1);

  finish_split(p, w, sm_m, sm_l, &sm_o[0][0], 256, heads_lo, heads_hi, 0, D, cta_index(p), w.first_cta, w.nsplit,
               w.nsplit * (p.nq > 1 ? gridDim.z : gridDim.y), &sm_flag, sm_scratch);
}

}  // namespace

cudaError_t launch_generic_attention(const AttnParams& p, cudaStream_t s) {
  if (p.total_ctas <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  const int hb = (p.group + kGenHeads - 1) / kGenHeads;
  cfg.gridDim = p.nq > 1 ? dim3(p.nq, p.total_ctas, hb) : dim3(p.total_ctas, hb, 1);
  cfg.blockDim = dim3(kGenWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, generic_attn_kernel, p);
}

}  // namespace ol
