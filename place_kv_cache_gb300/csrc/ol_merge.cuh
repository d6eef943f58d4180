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
  float* m;       // [8] CTA state
  float* l;       // [8]
  float* cm;      // [8] cluster state
  float* cl;      // [8]
  float* cw;      // [16][8] cluster weights
  float* cwl;     // [16][8] weighted cluster sums
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

// Merge `nstates` states (state s has O at state_o(s)) into the CTA state
// `merged` ([8][kOStride]) and ms.m / ms.l, then finish: with p.cluster == 1
// through finish_split; otherwise through the cluster merge (CTA rank r
// merges dims [r*128/CS, (r+1)*128/CS) of every head from all CS CTAs) and
// then finish_split on those dims. Every thread of every CTA of the cluster
// must call it (it contains cluster barriers when p.cluster > 1).
template <typename StateO>
__device__ __forceinline__ void merge_and_finish(const AttnParams& p, const Work& w, int nstates, StateO state_o,
                                                 float* merged, float* cmerged, const MergeScratch& ms) {
  const int G = p.group;
  const int CS = p.cluster;
  __syncthreads();
  if (threadIdx.x < 8) {
    const int j = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < nstates; ++s) M = fmaxf(M, ms.wm[s * 8 + j]);
    float L = 0.f;
    if (M != -INFINITY)
      for (int s = 0; s < nstates; ++s) {
        const float mw = ms.wm[s * 8 + j];
        if (mw != -INFINITY) L += ms.wl[s * 8 + j] * fast_exp2(mw - M);
      }
    ms.m[j] = M;
    ms.l[j] = L;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * 128; idx += blockDim.x) {
    const int j = idx >> 7, d = idx & 127;
    const float M = ms.m[j];
    float acc = 0.f;
    if (M != -INFINITY)
      for (int s = 0; s < nstates; ++s) {
        const float mw = ms.wm[s * 8 + j];
        if (mw != -INFINITY) acc += state_o(s)[j * kOStride + d] * fast_exp2(mw - M);
      }
    merged[j * kOStride + d] = acc;
  }
  __syncthreads();
  if (CS == 1) {
    if (!w.valid) return;
    finish_split(p, w, ms.m, ms.l, merged, kOStride, 0, G, 0, 128, blockIdx.x, w.first_cta, w.nsplit, w.nsplit,
                 ms.flag, ms.scr);
    return;
  }
  // Cluster merge: after a cluster barrier every CTA reads the CS (m, l) pairs
  // of each head (one remote load per thread) and merges its slice of dims
  // from the CS CTAs' `merged` with independent remote loads.
  cluster_sync();
  const uint32_t rank = cluster_ctarank();
  const int dspan = 128 / CS, d0 = (int)rank * dspan;
  if (threadIdx.x < CS * 8) {
    const int q = threadIdx.x >> 3, j = threadIdx.x & 7;
    ms.cw[threadIdx.x] = ld_shared_cluster(map_shared_rank(smem_u32(ms.m + j), q));
    ms.cwl[threadIdx.x] = ld_shared_cluster(map_shared_rank(smem_u32(ms.l + j), q));
  }
  __syncthreads();
  if (threadIdx.x < 8) {
    float M = -INFINITY;
    for (int q = 0; q < CS; ++q) M = fmaxf(M, ms.cw[q * 8 + threadIdx.x]);
    ms.cm[threadIdx.x] = M;
  }
  __syncthreads();
  if (threadIdx.x < CS * 8) {  // weights 2^(m_q - M), zero for empty splits
    const float M = ms.cm[threadIdx.x & 7], mq = ms.cw[threadIdx.x];
    const float wq = (M == -INFINITY || mq == -INFINITY) ? 0.f : fast_exp2(mq - M);
    ms.cw[threadIdx.x] = wq;
    ms.cwl[threadIdx.x] *= wq;
  }
  __syncthreads();
  if (threadIdx.x < 8) {
    float L = 0.f;
    for (int q = 0; q < CS; ++q) L += ms.cwl[q * 8 + threadIdx.x];
    ms.cl[threadIdx.x] = L;
  }
  for (int idx = threadIdx.x; idx < G * dspan; idx += blockDim.x) {
    const int j = idx / dspan, d = d0 + idx % dspan;
    const uint32_t local = smem_u32(merged + j * kOStride + d);
    float acc = 0.f;
#pragma unroll 4
    for (int q = 0; q < CS; ++q) acc += ld_shared_cluster(map_shared_rank(local, q)) * ms.cw[q * 8 + j];
    cmerged[j * dspan + (d - d0)] = acc;
  }
  cluster_sync();  // every remote read is done before any CTA of the cluster exits
  if (!w.valid) return;
  finish_split(p, w, ms.cm, ms.cl, cmerged, dspan, 0, G, d0, d0 + dspan, (int)(blockIdx.x / CS), w.first_cta / CS,
               w.nsplit / CS, w.nsplit, ms.flag, ms.scr);
}

}  // namespace ol
