// ol_merge.cuh -- the end of a tensor-core decode CTA, shared by the bf16 and
// INT4 kernels: per-warp online-softmax states -> CTA state -> (optionally)
// cluster state through distributed shared memory -> y or a split-K partial.
#pragma once

#include "ol_common.cuh"

namespace ol {

constexpr int kOStride = 132;  // fp32 row stride of an [8 heads][128 dims] state in shared memory

// Shared-memory scratch of the merge (all small, fixed size).
struct MergeScratch {
  float* wm;      // [nstates][8] per-state maxima (log2 domain)
  float* wl;      // [nstates][8] per-state sums
  float* wt;      // [nstates][8] per-state weights 2^(m_s - M)
  float* m;       // [8] CTA state
  float* l;       // [8]
  float* cm;      // [8] cluster state
  float* cl;      // [8]
  float* cw;      // [16][8] cluster weights
  float* recv_o;  // [CS][8][128/CS] slices pushed by the cluster's CTAs (1024 floats)
  float* recv_m;  // [CS][8] their maxima
  float* recv_l;  // [CS][8] their sums
  float* scr;     // [16] final-merge scratch
  int* flag;
};

// A warp's online-softmax state after its token loop, as the m16n8k16 O^T
// accumulator fragments plus (m, l) for the lane's two heads 2(lane%4), +1; l
// is summed over the warp here. Fragment o[mt] row r (r = lane/4 or lane/4+8)
// holds dimension 16mt + r, or with INT4_DIMS the INT4 kernel's order:
// mt = 2b + h, row lane/4 -> 32b + 4(lane/4) + 2h, row lane/4+8 -> that + 1.
// Written to `so` ([8][kOStride] fp32) and wm/wl[idx].
template <bool INT4_DIMS = false>
__device__ __forceinline__ void store_warp_state(float* so, const MergeScratch& ms, int idx, const float (&o)[8][4],
                                                 float m0, float m1, float l0, float l1) {
  const int lane = threadIdx.x & 31, c = lane & 3, n = lane >> 2;
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int da = INT4_DIMS ? 32 * (mt >> 1) + 4 * n + 2 * (mt & 1) : 16 * mt + n;
    const int db = INT4_DIMS ? da + 1 : da + 8;
    so[(2 * c) * kOStride + da] = o[mt][0];
    so[(2 * c + 1) * kOStride + da] = o[mt][1];
    so[(2 * c) * kOStride + db] = o[mt][2];
    so[(2 * c + 1) * kOStride + db] = o[mt][3];
  }
  if (n == 0) {
    ms.wm[idx * 8 + 2 * c] = m0;
    ms.wm[idx * 8 + 2 * c + 1] = m1;
    ms.wl[idx * 8 + 2 * c] = l0;
    ms.wl[idx * 8 + 2 * c + 1] = l1;
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ void st_shared_cluster(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_shared_cluster_v4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

// Merge `nstates` (<= 32) states (state s has O at state_o(s)) into the CTA
// state and finish. Weights 2^(m_s - M) are formed once per (state, head).
//   p.cluster == 1: the CTA state goes to `merged` ([8][kOStride]) and
//     finish_split.
//   p.cluster == CS > 1: the CTAs of a cluster hold consecutive splits of one
//     (row, kv head); CTA r owns dims [r*128/CS, (r+1)*128/CS). Each CTA pushes
//     its state straight into the owners' receive buffers (remote shared-memory
//     stores), one cluster barrier makes them visible, and every CTA merges its
//     own slice from local shared memory. No remote loads, one barrier; after
//     the barrier a CTA touches only its own shared memory and may exit.
// Every thread of every CTA of the cluster must call it.
template <typename StateO>
__device__ __forceinline__ void merge_and_finish(const AttnParams& p, const Work& w, int nstates, StateO state_o,
                                                 float* merged, float* cmerged, const MergeScratch& ms,
                                                 int zs = -1) {
  const int G = state_cols(p);  // state columns: the heads, or (query token, head) pairs
  const int CS = p.cluster;
  __syncthreads();
  if (threadIdx.x < 8) {  // one thread per head: maximum, weights 2^(m_s - M), sum
    const int j = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < nstates; ++s) M = fmaxf(M, ms.wm[s * 8 + j]);
    float L = 0.f;
    for (int s = 0; s < nstates; ++s) {
      const float mw = ms.wm[s * 8 + j];
      const float wt = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
      ms.wt[s * 8 + j] = wt;
      L += wt * ms.wl[s * 8 + j];
    }
    ms.m[j] = M;
    ms.l[j] = L;
  }
  __syncthreads();
  const uint32_t rank = CS > 1 ? cluster_ctarank() : 0;
  const int dspan = 128 / CS;
  if (CS > 1 && threadIdx.x < CS * 8) {  // (m, l) of head j to CTA q
    const int q = threadIdx.x >> 3, j = threadIdx.x & 7;
    st_shared_cluster(map_shared_rank(smem_u32(ms.recv_m + rank * 8 + j), q), ms.m[j]);
    st_shared_cluster(map_shared_rank(smem_u32(ms.recv_l + rank * 8 + j), q), ms.l[j]);
  }
  for (int idx = threadIdx.x; idx < G * 32; idx += blockDim.x) {
    const int j = idx >> 5, d = (idx & 31) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < nstates; ++s) {
      const float wt = ms.wt[s * 8 + j];
      if (wt != 0.f) {
        const float4 v = *reinterpret_cast<const float4*>(state_o(s) + j * kOStride + d);
        acc.x += wt * v.x;
        acc.y += wt * v.y;
        acc.z += wt * v.z;
        acc.w += wt * v.w;
      }
    }
    if (CS == 1) {
      *reinterpret_cast<float4*>(merged + j * kOStride + d) = acc;
    } else {
      const int owner = d / dspan;
      const uint32_t dst = smem_u32(ms.recv_o + (rank * 8 + j) * dspan + (d - owner * dspan));
      st_shared_cluster_v4(map_shared_rank(dst, owner), acc);
    }
  }
  if (CS == 1) {
    __syncthreads();
    if (!w.valid) return;
    finish_split(p, w, ms.m, ms.l, merged, kOStride, 0, G, 0, 128, w.slot, w.first_cta, w.nsplit, w.nsplit,
                 ms.flag, ms.scr, zs);
    return;
  }
  cluster_sync();  // every push of every CTA of the cluster is visible
  const int d0 = (int)rank * dspan;
  if (threadIdx.x < 8) {
    const int j = threadIdx.x;
    float M = -INFINITY;
    for (int q = 0; q < CS; ++q) M = fmaxf(M, ms.recv_m[q * 8 + j]);
    float L = 0.f;
    for (int q = 0; q < CS; ++q) {
      const float mq = ms.recv_m[q * 8 + j];
      const float wq = (mq == -INFINITY) ? 0.f : fast_exp2(mq - M);
      ms.cw[q * 8 + j] = wq;
      L += wq * ms.recv_l[q * 8 + j];
    }
    ms.cm[j] = M;
    ms.cl[j] = L;
  }
  __syncthreads();
  const int nd4 = dspan / 4;
  for (int idx = threadIdx.x; idx < G * nd4; idx += blockDim.x) {
    const int j = idx / nd4, dd = (idx % nd4) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < CS; ++q) {
      const float wq = ms.cw[q * 8 + j];
      const float4 v = *reinterpret_cast<const float4*>(ms.recv_o + (q * 8 + j) * dspan + dd);
      acc.x += wq * v.x;
      acc.y += wq * v.y;
      acc.z += wq * v.z;
      acc.w += wq * v.w;
    }
    *reinterpret_cast<float4*>(cmerged + j * dspan + dd) = acc;
  }
  __syncthreads();
  if (!w.valid) return;
  finish_split(p, w, ms.cm, ms.cl, cmerged, dspan, 0, G, d0, d0 + dspan, cta_index(p) / CS, w.first_cta / CS,
               w.nsplit / CS, w.nsplit, ms.flag, ms.scr, zs);
}

}  // namespace ol
