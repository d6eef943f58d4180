// ol_merge.cuh -- the end of a tensor-core decode CTA, shared by the bf16 and
// INT4 kernels: per-warp online-softmax states -> CTA state -> (optionally)
// cluster state through distributed shared memory -> y or a split-K partial.
#pragma once

#include "ol_common.cuh"

// Phase stamps of the timing build (see ol_fast_bf16.cu); no code otherwise.
#ifndef OL_STAMP
#define OL_STAMP(ph)
#define OL_STAMP_AFTER(ph, reg)
#define OL_STAMP_BEGIN(on)
#define OL_STAMP_END()
#endif

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

// The last level of a cluster merge when the cluster covers its (row, kv head)
// alone: thread (column j, 4 dims) of this CTA's slice [rank*128/CS, +128/CS)
// forms M = max_q m_q, the weights 2^(m_q - M) and L = sum_q l_q 2^(m_q - M)
// over the CS received states and stores y = sum_q o_q 2^(m_q - M) / L.
template <int CS>
__device__ __forceinline__ void cluster_store_y(const AttnParams& p, const Work& w, const MergeScratch& ms, int G,
                                                int zs) {
  constexpr int dspan = 128 / CS, nd4 = dspan / 4;
  const int d0 = (int)cluster_ctarank() * dspan;
  if (zs < 0) zs = query_index(p);
  const int D = p.head_dim, Gq = p.group;
  const int nq = p.nq > 1 ? p.nq : 1, z0 = slice_first(p, zs), c_live = Gq * slice_tokens(p, zs);
  const size_t head_base = (size_t)w.b * p.q_heads + (size_t)w.g * Gq;
  for (int idx = threadIdx.x; idx < G * nd4; idx += blockDim.x) {
    const int j = idx / nd4, dd = (idx % nd4) * 4;
    float mq[CS], t[CS];
#pragma unroll
    for (int q = 0; q < CS; ++q) t[q] = mq[q] = ms.recv_m[q * 8 + j];
#pragma unroll
    for (int h = CS / 2; h >= 1; h >>= 1)  // the maximum as a tree
#pragma unroll
      for (int q = 0; q < h; ++q) t[q] = fmaxf(t[q], t[q + h]);
    const float M = t[0];
    // two partial sums per quantity: half the dependent chain
    float L2[2] = {0.f, 0.f};
    float4 acc2[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
#pragma unroll
    for (int q = 0; q < CS; ++q) {
      const float wq = (mq[q] == -INFINITY) ? 0.f : fast_exp2(mq[q] - M);
      L2[q & 1] += wq * ms.recv_l[q * 8 + j];
      const float4 v = *reinterpret_cast<const float4*>(ms.recv_o + (q * 8 + j) * dspan + dd);
      acc2[q & 1].x += wq * v.x;
      acc2[q & 1].y += wq * v.y;
      acc2[q & 1].z += wq * v.z;
      acc2[q & 1].w += wq * v.w;
    }
    const float L = L2[0] + L2[1];
    const float4 acc = make_float4(acc2[0].x + acc2[1].x, acc2[0].y + acc2[1].y, acc2[0].z + acc2[1].z,
                                   acc2[0].w + acc2[1].w);
    if (j >= c_live) continue;
    const size_t o = (nq == 1 ? (head_base + j) : ((head_base + j % Gq) * nq + z0 + j / Gq)) * D + d0 + dd;
    const float rl = L > 0.f ? 1.f / L : 0.f;  // one division, four products
    const float y0 = acc.x * rl, y1 = acc.y * rl, y2 = acc.z * rl, y3 = acc.w * rl;
    if (p.out_dtype == OL_F32) {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + o) = make_float4(y0, y1, y2, y3);
    } else {
      *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.out) + o) =
          make_uint2(pack_bf16x2(y0, y1), pack_bf16x2(y2, y3));
    }
  }
}

// Merge `nstates` (<= 32) states (state s has O at state_o(s)) into the CTA
// state and finish.
//   CTA level: thread (head j, 8 dims d..d+7) forms head j's maximum M over the
//     states, the weights 2^(m_s - M) and L = sum_s l_s 2^(m_s - M) in its own
//     registers (every thread of a head recomputes them from shared memory: no
//     barrier between the reduction and its use), then its 8 dims of
//     sum_s o_s 2^(m_s - M).
//   p.cluster == 1: the CTA state goes to `merged` ([8][kOStride]) and
//     finish_split.
//   p.cluster == CS > 1: the CTAs of a cluster hold consecutive splits of one
//     (row, kv head); CTA r owns dims [r*128/CS, (r+1)*128/CS). Each CTA pushes
//     its state straight into the owners' receive buffers (remote shared-memory
//     stores), one cluster barrier makes them visible, and every CTA merges its
//     own slice from local shared memory. No remote loads, one barrier; after
//     the barrier a CTA touches only its own shared memory and may exit. When
//     the cluster covers its (row, kv head) alone, thread (head j, 4 dims)
//     forms the merge weights in registers and stores y directly (no further
//     barrier); otherwise the cluster state goes to finish_split.
// NS > 0: the caller passes exactly NS states, every one with its O written
// (zero for a state that saw no visible token), so the CTA level needs no
// data-dependent branch and the loads of all states issue together; NS = 0:
// nstates is known only at run time, and a state of weight 0 is skipped.
// Every thread of every CTA of the cluster must call it.
template <int NS = 0, typename StateO>
__device__ __forceinline__ void merge_and_finish(const AttnParams& p, const Work& w, int nstates, StateO state_o,
                                                 float* merged, float* cmerged, const MergeScratch& ms,
                                                 int zs = -1) {
  const int G = state_cols(p);  // state columns: the heads, or (query token, head) pairs
  const int CS = p.cluster;
  __syncthreads();
  OL_STAMP(OL_PH_ALL_TILES);
  const uint32_t rank = CS > 1 ? cluster_ctarank() : 0;
  const int dspan = 128 / CS;
  for (int idx = threadIdx.x; idx < G * 16; idx += blockDim.x) {
    const int j = idx >> 4, d = (idx & 15) * 8;
    float M = -INFINITY;
    float L = 0.f;
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
    // state s's 8 dims of head j, weighted
    auto add = [&](int s, float wt) {
      const float4 v0 = *reinterpret_cast<const float4*>(state_o(s) + j * kOStride + d);
      const float4 v1 = *reinterpret_cast<const float4*>(state_o(s) + j * kOStride + d + 4);
      a0.x += wt * v0.x;
      a0.y += wt * v0.y;
      a0.z += wt * v0.z;
      a0.w += wt * v0.w;
      a1.x += wt * v1.x;
      a1.y += wt * v1.y;
      a1.z += wt * v1.z;
      a1.w += wt * v1.w;
    };
    if constexpr (NS > 0) {
      float mw[NS];
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        mw[s] = ms.wm[s * 8 + j];
        M = fmaxf(M, mw[s]);
      }
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        const float wt = (mw[s] == -INFINITY) ? 0.f : fast_exp2(mw[s] - M);
        L += wt * ms.wl[s * 8 + j];
        add(s, wt);
      }
    } else {
#pragma unroll 8
      for (int s = 0; s < nstates; ++s) M = fmaxf(M, ms.wm[s * 8 + j]);
#pragma unroll 8
      for (int s = 0; s < nstates; ++s) {
        const float mw = ms.wm[s * 8 + j];
        const float wt = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
        L += wt * ms.wl[s * 8 + j];
        if (wt != 0.f) add(s, wt);
      }
    }
    if (CS == 1) {
      *reinterpret_cast<float4*>(merged + j * kOStride + d) = a0;
      *reinterpret_cast<float4*>(merged + j * kOStride + d + 4) = a1;
      if (d == 0) {
        ms.m[j] = M;
        ms.l[j] = L;
      }
    } else {
      const int owner = d / dspan, off = d - owner * dspan;
      const uint32_t dst = smem_u32(ms.recv_o + (rank * 8 + j) * dspan + off);
      st_shared_cluster_v4(map_shared_rank(dst, owner), a0);
      st_shared_cluster_v4(map_shared_rank(dst + 16, owner), a1);
      if (off == 0) {  // the owner of these dims also needs this CTA's (m, l) of head j
        st_shared_cluster(map_shared_rank(smem_u32(ms.recv_m + rank * 8 + j), owner), M);
        st_shared_cluster(map_shared_rank(smem_u32(ms.recv_l + rank * 8 + j), owner), L);
      }
    }
  }
  if (CS == 1) {
    __syncthreads();
    if (!w.valid) return;
    finish_split(p, w, ms.m, ms.l, merged, kOStride, 0, G, 0, 128, w.slot, w.first_cta, w.nsplit, w.nsplit,
                 ms.flag, ms.scr, zs);
    return;
  }
  OL_STAMP(OL_PH_CTA_MERGED);
  cluster_sync();  // every push of every CTA of the cluster is visible
  OL_STAMP(OL_PH_CLUSTER);
  const int d0 = (int)rank * dspan;
  const int nd4 = dspan / 4;
  if (w.nsplit == CS) {
    // the cluster is the whole (row, kv head): y for this CTA's dims, straight from registers
    if (!w.valid) return;
    switch (CS) {  // a compile-time source count lets every source's loads issue together
      case 16: cluster_store_y<16>(p, w, ms, G, zs); return;
      case 8: cluster_store_y<8>(p, w, ms, G, zs); return;
      case 4: cluster_store_y<4>(p, w, ms, G, zs); return;
      default: cluster_store_y<2>(p, w, ms, G, zs); return;
    }
  }
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
