// ol_hpaged.cuh -- element codecs of the heterogeneous paged cache: every page
// stores K and V in its own format (dense FLOAT / FLOAT16 / BFLOAT16, or affine
// INT8 / UINT8 / INT4 / UINT4 / INT2 / UINT2 with one scalar scale and zero
// point per page and plane). Encoding is QuantizeLinear in IEEE fp32 (true
// division, round half to even, saturation to the code range); decoding is
// (code - zero_point) * scale in fp32. Four- and two-bit codes pack two and
// four per byte, least-significant bits first.
#pragma once

#include "ol_common.cuh"

namespace ol {

// Byte address of the row (head h, page slot s) of plane `plane` of page `page`.
__device__ __forceinline__ uint8_t* hp_row(uint8_t* pool, int kv_heads, int S, int D, int page, int plane, int h,
                                           int s, int f) {
  const size_t plane_bytes = (size_t)kv_heads * S * D * 4;
  return pool + (size_t)page * 2 * plane_bytes + (size_t)plane * plane_bytes + ((size_t)h * S + s) * fmt_row_bytes(f, D);
}

// Element d of a row, decoded to fp32.
__device__ __forceinline__ float hp_decode(const uint8_t* row, int d, const ol_plane_format& pf) {
  switch (pf.format) {
    case OL_FMT_F32: return reinterpret_cast<const float*>(row)[d];
    case OL_FMT_F16: return fp16_bits_to_float(reinterpret_cast<const uint16_t*>(row)[d]);
    case OL_FMT_BF16: return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(row)[d]);
    default: break;
  }
  const int bits = fmt_bits(pf.format);
  int code;
  if (bits == 8) {
    code = row[d];
  } else {
    code = (row[(size_t)d * bits / 8] >> ((d * bits) & 7)) & ((1 << bits) - 1);
  }
  if (fmt_signed(pf.format) && code >= (1 << (bits - 1))) code -= 1 << bits;
  return (float)(code - pf.zero_point) * pf.scale;
}

// QuantizeLinear of one value to a code of an affine format (as unsigned bits).
__device__ __forceinline__ unsigned hp_code(float x, const ol_plane_format& pf) {
  float r = rintf(__fdiv_rn(x, pf.scale)) + (float)pf.zero_point;
  r = fminf(fmaxf(r, (float)fmt_qmin(pf.format)), (float)fmt_qmax(pf.format));
  return (unsigned)(int)r & ((1u << fmt_bits(pf.format)) - 1u);
}

// One warp encodes a row of D fp32 values (element d from value(d)) into `row`.
template <typename ValueAt>
__device__ __forceinline__ void hp_encode_row_warp(ValueAt value, int D, const ol_plane_format& pf, uint8_t* row) {
  const int lane = threadIdx.x & 31;
  const int f = pf.format;
  if (f == OL_FMT_F32) {
    for (int d = lane; d < D; d += 32) reinterpret_cast<float*>(row)[d] = value(d);
  } else if (f == OL_FMT_F16) {
    for (int d = lane; d < D; d += 32) {
      __half h = __float2half_rn(value(d));
      reinterpret_cast<uint16_t*>(row)[d] = *reinterpret_cast<uint16_t*>(&h);
    }
  } else if (f == OL_FMT_BF16) {
    for (int d = lane; d < D; d += 32) reinterpret_cast<uint16_t*>(row)[d] = float_to_bf16_bits(value(d));
  } else {
    const int bits = fmt_bits(f), per = 8 / bits;  // codes per byte
    const int nbytes = D * bits / 8;
    for (int j = lane; j < nbytes; j += 32) {
      unsigned byte = 0;
      for (int k = 0; k < per; ++k) byte |= hp_code(value(j * per + k), pf) << (k * bits);
      row[j] = (uint8_t)byte;
    }
  }
}

}  // namespace ol
