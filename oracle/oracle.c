/*
 * oracle.c -- plain, slow CPU oracle for the decode step over a caller-owned
 * KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file: it exists so the CUDA kernels can be checked against an
 * independent statement of what they compute. It shares no code, header,
 * table or constant with the CUDA library.
 *
 * Every function writes out the plain definition:
 *   - CacheUpdate: copy `values` into the cache rows starting at `position`,
 *     reject position + new_len > capacity, write nothing else
 *     (page "Mutable execution cache", sections Value model, Model example,
 *     Runtime contract).
 *   - PagedCacheUpdate: the same, through a block table of fixed-size pages
 *     (same page, sections Heterogeneous paged cache and ONNX Runtime GenAI).
 *   - Decode attention: for each query head h of row b, kv head g = h / G,
 *     scores s_t = scale * q . k_t over the visible tokens, a plain two-pass
 *     softmax in fp64 and y = sum_t w_t v_t (page "Persistent input/output
 *     feedback", section Optional heterogeneous paged KV, kernel paragraphs on
 *     causal masking, left_window_size and grouped-query attention).
 *   - INT4 blockwise affine: per block of 32 elements one fp16 scale and one
 *     uint4 zero point, code = saturate(round_half_even(x / scale) + zp),
 *     two codes per byte with the first in the low nibble, reconstruction
 *     (code - zp) * scale (page "Custom, quantized, and persistent values",
 *     section Struct types and byte-encodable layouts; page "Persistent
 *     input/output feedback", rounding and tolerance paragraph).
 *
 * Precision: attention in fp64; quantization decisions in IEEE fp32 (true
 * division, round-half-even, no contraction) with the scale rounded to fp16,
 * the precision the quantized format itself fixes. Compile with
 * -ffp-contract=off and without fast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum {
  ORC_OK = 0,
  ORC_ERR_CAPACITY = 4,
  ORC_ERR_SHAPE = 5,
  ORC_ERR_PAGE = 13,
  ORC_ERR_ALLOC = 20
};
enum { ORC_Q_DYNAMIC = 0, ORC_Q_FIXED = 1 };

/* ---------------------------------------------------------------- scalars */

static double bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static float bf16_to_float(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static double fp16_bits_to_double(uint16_t bits) {
  _Float16 h;
  memcpy(&h, &bits, sizeof h);
  return (double)h;
}

static uint16_t float_to_fp16_bits(float f) {
  _Float16 h = (_Float16)f; /* IEEE conversion, round to nearest even */
  uint16_t bits;
  memcpy(&bits, &h, sizeof bits);
  return bits;
}

static size_t elt_size(int dtype) { return dtype == ORC_F32 ? 4u : 2u; }

static double load_elem(const void* base, int dtype, size_t i) {
  if (dtype == ORC_F32) return (double)((const float*)base)[i];
  return bf16_to_double(((const uint16_t*)base)[i]);
}

/* fp16 bits -> double, exposed for tests */
double orc_fp16_to_double(uint16_t bits) { return fp16_bits_to_double(bits); }
uint16_t orc_float_to_fp16(float f) { return float_to_fp16_bits(f); }

/* ------------------------------------------------------------- visibility */

/*
 * Causal decode visibility. The query sits at position p = n - 1 and sees
 * [0, p]; with a left window w >= 0 it sees the w preceding tokens and itself,
 * [max(0, p - w), p]; w < 0 means unbounded (left_window_size = -1).
 * Returns the number of visible tokens; [*lo, *hi) is the visible range.
 */
int orc_visible_range(int n, int window, int* lo, int* hi) {
  if (n <= 0) {
    *lo = 0;
    *hi = 0;
    return 0;
  }
  int p = n - 1;
  *hi = n;
  if (window < 0)
    *lo = 0;
  else
    *lo = (p - window > 0) ? p - window : 0;
  return *hi - *lo;
}

/* ------------------------------------------------------------- attention */

/*
 * Softmax attention of one query over n materialized tokens, in fp64:
 *   s_t = scale * sum_d q_d k_{t,d};  w_t = exp(s_t - max s) / sum exp(s - max s);
 *   y_d = sum_t w_t v_{t,d}.
 * n == 0 gives y = 0 (the empty sum).
 */
static int attend_one(const double* q, const double* K, const double* V, int n, int D,
                      double scale, double* y) {
  for (int d = 0; d < D; ++d) y[d] = 0.0;
  if (n == 0) return ORC_OK;
  double* s = (double*)malloc((size_t)n * sizeof(double));
  if (!s) return ORC_ERR_ALLOC;
  double m = -INFINITY;
  for (int t = 0; t < n; ++t) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += q[d] * K[(size_t)t * D + d];
    s[t] = scale * acc;
    if (s[t] > m) m = s[t];
  }
  double z = 0.0;
  for (int t = 0; t < n; ++t) {
    s[t] = exp(s[t] - m);
    z += s[t];
  }
  for (int t = 0; t < n; ++t) {
    double w = s[t] / z;
    for (int d = 0; d < D; ++d) y[d] += w * V[(size_t)t * D + d];
  }
  free(s);
  return ORC_OK;
}

/* Attend every query head of one (row, kv head) group to materialized K/V. */
static int attend_group(const void* q, int q_dtype, int Hq, int G, int b, int g, int D,
                        const double* K, const double* V, int n, double scale, double* out) {
  double* qv = (double*)malloc((size_t)D * sizeof(double));
  if (!qv) return ORC_ERR_ALLOC;
  int rc = ORC_OK;
  for (int j = 0; j < G && rc == ORC_OK; ++j) {
    int h = g * G + j;
    size_t qbase = ((size_t)b * Hq + h) * D;
    for (int d = 0; d < D; ++d) qv[d] = load_elem(q, q_dtype, qbase + d);
    rc = attend_one(qv, K, V, n, D, scale, out + qbase);
  }
  free(qv);
  return rc;
}

/*
 * Decode attention over a contiguous cache [2, B, Hkv, C, D] (K plane 0,
 * V plane 1). q is [B, Hq, D]; out is [B, Hq, D] fp64. lens[b] counts the
 * attended tokens of row b (0 <= lens[b] <= C).
 */
int orc_decode_attention(const void* q, int q_dtype, int Hq, const void* cache, int c_dtype,
                         int B, int Hkv, int C, int D, const int32_t* lens, double scale,
                         int window, double* out) {
  if (B < 0 || Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0 || D <= 0 || C < 0) return ORC_ERR_SHAPE;
  for (int b = 0; b < B; ++b)
    if (lens[b] < 0 || lens[b] > C) return ORC_ERR_CAPACITY;
  int G = Hq / Hkv;
  double* K = (double*)malloc(((size_t)C + 1) * D * sizeof(double));
  double* V = (double*)malloc(((size_t)C + 1) * D * sizeof(double));
  if (!K || !V) {
    free(K);
    free(V);
    return ORC_ERR_ALLOC;
  }
  int rc = ORC_OK;
  for (int b = 0; b < B && rc == ORC_OK; ++b) {
    int lo, hi;
    int n = orc_visible_range(lens[b], window, &lo, &hi);
    for (int g = 0; g < Hkv && rc == ORC_OK; ++g) {
      for (int t = 0; t < n; ++t) {
        size_t kbase = ((((size_t)0 * B + b) * Hkv + g) * C + (lo + t)) * D;
        size_t vbase = ((((size_t)1 * B + b) * Hkv + g) * C + (lo + t)) * D;
        for (int d = 0; d < D; ++d) {
          K[(size_t)t * D + d] = load_elem(cache, c_dtype, kbase + d);
          V[(size_t)t * D + d] = load_elem(cache, c_dtype, vbase + d);
        }
      }
      rc = attend_group(q, q_dtype, Hq, G, b, g, D, K, V, n, scale, out);
    }
  }
  free(K);
  free(V);
  return rc;
}

/*
 * Decode attention over a paged pool [2, P, Hkv, S, D] with block table
 * [B, M]: logical token t of row b is slot t % S of page block_table[b][t / S].
 * Defined as contiguous attention on the gathered logical sequence.
 */
int orc_paged_attention(const void* q, int q_dtype, int Hq, const void* pool, int c_dtype,
                        int P, int Hkv, int S, int D, const int32_t* block_table, int M, int B,
                        const int32_t* lens, double scale, int window, double* out) {
  if (B < 0 || Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0 || D <= 0 || S <= 0 || M < 0)
    return ORC_ERR_SHAPE;
  long long cap = (long long)M * S;
  for (int b = 0; b < B; ++b) {
    if (lens[b] < 0 || lens[b] > cap) return ORC_ERR_CAPACITY;
    for (int t = 0; t < lens[b]; ++t) {
      int page = block_table[(size_t)b * M + t / S];
      if (page < 0 || page >= P) return ORC_ERR_PAGE;
    }
  }
  int G = Hq / Hkv;
  double* K = (double*)malloc(((size_t)cap + 1) * D * sizeof(double));
  double* V = (double*)malloc(((size_t)cap + 1) * D * sizeof(double));
  if (!K || !V) {
    free(K);
    free(V);
    return ORC_ERR_ALLOC;
  }
  int rc = ORC_OK;
  for (int b = 0; b < B && rc == ORC_OK; ++b) {
    int lo, hi;
    int n = orc_visible_range(lens[b], window, &lo, &hi);
    for (int g = 0; g < Hkv && rc == ORC_OK; ++g) {
      for (int t = 0; t < n; ++t) {
        int logical = lo + t;
        int page = block_table[(size_t)b * M + logical / S];
        int slot = logical % S;
        size_t kbase = ((((size_t)0 * P + page) * Hkv + g) * S + slot) * D;
        size_t vbase = ((((size_t)1 * P + page) * Hkv + g) * S + slot) * D;
        for (int d = 0; d < D; ++d) {
          K[(size_t)t * D + d] = load_elem(pool, c_dtype, kbase + d);
          V[(size_t)t * D + d] = load_elem(pool, c_dtype, vbase + d);
        }
      }
      rc = attend_group(q, q_dtype, Hq, G, b, g, D, K, V, n, scale, out);
    }
  }
  free(K);
  free(V);
  return rc;
}

/* ---------------------------------------------------------------- appends */

/*
 * CacheUpdate on a contiguous cache [2, B, H, C, D]: for k in {K, V}, every
 * row b and head h, cache[k][b][h][p_b + j] = values[k][b][h][j] for
 * j < new_len, where p_b = positions[b]. Rejects any row with
 * p_b < 0 or p_b + new_len > C before writing anything.
 */
int orc_cache_update(void* cache, int dtype, int B, int H, int C, int D, const void* values,
                     int new_len, const int32_t* positions) {
  if (B < 0 || H <= 0 || D <= 0 || C < 0 || new_len < 0) return ORC_ERR_SHAPE;
  for (int b = 0; b < B; ++b)
    if (positions[b] < 0 || (long long)positions[b] + new_len > C) return ORC_ERR_CAPACITY;
  size_t es = elt_size(dtype);
  for (int k = 0; k < 2; ++k)
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h)
        for (int j = 0; j < new_len; ++j) {
          size_t dst = ((((size_t)k * B + b) * H + h) * C + (positions[b] + j)) * D;
          size_t src = ((((size_t)k * B + b) * H + h) * new_len + j) * D;
          memcpy((char*)cache + dst * es, (const char*)values + src * es, (size_t)D * es);
        }
  return ORC_OK;
}

/*
 * PagedCacheUpdate on a pool [2, P, H, S, D] through block table [B, M]:
 * logical token p_b + j of row b goes to slot (p_b + j) % S of page
 * block_table[b][(p_b + j) / S]. Everything is validated before any write.
 */
int orc_paged_update(void* pool, int dtype, int P, int H, int S, int D, const int32_t* block_table,
                     int M, int B, const void* values, int new_len, const int32_t* positions) {
  if (B < 0 || H <= 0 || D <= 0 || S <= 0 || M < 0 || new_len < 0) return ORC_ERR_SHAPE;
  long long cap = (long long)M * S;
  for (int b = 0; b < B; ++b) {
    if (positions[b] < 0 || (long long)positions[b] + new_len > cap) return ORC_ERR_CAPACITY;
    for (int j = 0; j < new_len; ++j) {
      int t = positions[b] + j;
      int page = block_table[(size_t)b * M + t / S];
      if (page < 0 || page >= P) return ORC_ERR_PAGE;
    }
  }
  size_t es = elt_size(dtype);
  for (int k = 0; k < 2; ++k)
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h)
        for (int j = 0; j < new_len; ++j) {
          int t = positions[b] + j;
          int page = block_table[(size_t)b * M + t / S];
          size_t dst = ((((size_t)k * P + page) * H + h) * S + (t % S)) * D;
          size_t src = ((((size_t)k * B + b) * H + h) * new_len + j) * D;
          memcpy((char*)pool + dst * es, (const char*)values + src * es, (size_t)D * es);
        }
  return ORC_OK;
}

/* ------------------------------------------------------------------- INT4 */

/* Pack n 4-bit codes, first code in the low nibble; a final odd code leaves the high nibble zero. */
void orc_pack_u4(const uint8_t* codes, int n, uint8_t* out) {
  for (int i = 0; i < (n + 1) / 2; ++i) {
    uint8_t lo = codes[2 * i] & 0xF;
    uint8_t hi = (2 * i + 1 < n) ? (codes[2 * i + 1] & 0xF) : 0;
    out[i] = (uint8_t)(lo | (hi << 4));
  }
}

void orc_unpack_u4(const uint8_t* packed, int n, uint8_t* codes) {
  for (int i = 0; i < n; ++i) codes[i] = (i % 2 == 0) ? (packed[i / 2] & 0xF) : (packed[i / 2] >> 4);
}

/* saturate(round_half_even(v) + zp) to [0, 15], taken in fp32 */
static uint8_t quantize_one(float x, float scale, int zp) {
  float r = rintf(x / scale) + (float)zp;
  if (r < 0.0f) r = 0.0f;
  if (r > 15.0f) r = 15.0f;
  return (uint8_t)r;
}

/*
 * Quantize one block of 32 values to uint4 codes with one fp16 scale and one
 * uint4 zero point.
 *   fixed mode:   scale = fp16(fixed_scale), zp = fixed_zp (the selector's
 *                 scalar parameters, e.g. UINT4 0.25 / 8).
 *   dynamic mode: lo = min(0, min x), hi = max(0, max x),
 *                 scale = fp16((hi - lo) / 15) (1.0 if that is 0),
 *                 zp = saturate(round_half_even(-lo / scale)).
 * Codes always use the stored fp16 scale.
 */
static void quantize_block(const float* x, int n, int mode, float fixed_scale, int fixed_zp,
                           uint8_t* codes, uint16_t* scale_bits, uint8_t* zp_out) {
  float s;
  int zp;
  if (mode == ORC_Q_FIXED) {
    *scale_bits = float_to_fp16_bits(fixed_scale);
    s = (float)fp16_bits_to_double(*scale_bits);
    zp = fixed_zp;
  } else {
    float lo = 0.0f, hi = 0.0f;
    for (int i = 0; i < n; ++i) {
      if (x[i] < lo) lo = x[i];
      if (x[i] > hi) hi = x[i];
    }
    float s32 = (hi - lo) / 15.0f;
    *scale_bits = float_to_fp16_bits(s32);
    s = (float)fp16_bits_to_double(*scale_bits);
    if (s == 0.0f) {
      *scale_bits = float_to_fp16_bits(1.0f);
      s = 1.0f;
    }
    float z = rintf(-lo / s);
    if (z < 0.0f) z = 0.0f;
    if (z > 15.0f) z = 15.0f;
    zp = (int)z;
  }
  *zp_out = (uint8_t)zp;
  for (int i = 0; i < n; ++i) codes[i] = quantize_one(x[i], s, zp);
}

/*
 * Quantize one token's D bf16 values (D a multiple of 32) into the planar
 * INT4 row format: D/2 packed code bytes, D/32 fp16 scales, ceil(D/64) packed
 * zero-point bytes. Returns ORC_ERR_SHAPE if D is not a multiple of 32.
 */
int orc_int4_quantize_row(const uint16_t* x_bf16, int D, int mode, float fixed_scale, int fixed_zp,
                          uint8_t* codes_packed, uint16_t* scales, uint8_t* zps_packed) {
  if (D <= 0 || D % 32 != 0) return ORC_ERR_SHAPE;
  int nb = D / 32;
  uint8_t codes[32];
  uint8_t zp_unpacked[64];
  float xf[32];
  if (nb > 64) return ORC_ERR_SHAPE;
  for (int blk = 0; blk < nb; ++blk) {
    for (int i = 0; i < 32; ++i) xf[i] = bf16_to_float(x_bf16[blk * 32 + i]);
    quantize_block(xf, 32, mode, fixed_scale, fixed_zp, codes, &scales[blk], &zp_unpacked[blk]);
    orc_pack_u4(codes, 32, codes_packed + blk * 16);
  }
  orc_pack_u4(zp_unpacked, nb, zps_packed);
  return ORC_OK;
}

/* Reconstruct one token's D values: (code - zp) * scale, exact in fp64. */
int orc_int4_dequantize_row(const uint8_t* codes_packed, const uint16_t* scales,
                            const uint8_t* zps_packed, int D, double* out) {
  if (D <= 0 || D % 32 != 0) return ORC_ERR_SHAPE;
  int nb = D / 32;
  for (int d = 0; d < D; ++d) {
    int blk = d / 32;
    int code = (d % 2 == 0) ? (codes_packed[d / 2] & 0xF) : (codes_packed[d / 2] >> 4);
    int zp = (blk % 2 == 0) ? (zps_packed[blk / 2] & 0xF) : (zps_packed[blk / 2] >> 4);
    out[d] = (double)(code - zp) * fp16_bits_to_double(scales[blk]);
  }
  (void)nb;
  return ORC_OK;
}

/* bytes per token row of each INT4 plane */
static int codes_row(int D) { return D / 2; }
static int scales_row(int D) { return D / 32; }
static int zps_row(int D) { return (D / 32 + 1) / 2; }

/*
 * INT4 append: quantize values [2, B, H, new_len, D] (bf16) and write them at
 * rows positions[b] .. positions[b] + new_len - 1 of the planes
 *   codes  [2, B, H, C, D/2]   uint8
 *   scales [2, B, H, C, D/32]  fp16 bits
 *   zps    [2, B, H, C, ceil(D/64)] uint8
 */
int orc_int4_append(uint8_t* codes, uint16_t* scales, uint8_t* zps, int B, int H, int C, int D,
                    const uint16_t* values, int new_len, const int32_t* positions, int mode,
                    float fixed_scale, int fixed_zp) {
  if (B < 0 || H <= 0 || D <= 0 || D % 32 != 0 || new_len < 0) return ORC_ERR_SHAPE;
  for (int b = 0; b < B; ++b)
    if (positions[b] < 0 || (long long)positions[b] + new_len > C) return ORC_ERR_CAPACITY;
  int cr = codes_row(D), sr = scales_row(D), zr = zps_row(D);
  for (int k = 0; k < 2; ++k)
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h)
        for (int j = 0; j < new_len; ++j) {
          size_t row = (((size_t)k * B + b) * H + h) * C + (positions[b] + j);
          size_t src = ((((size_t)k * B + b) * H + h) * new_len + j) * D;
          int rc = orc_int4_quantize_row(values + src, D, mode, fixed_scale, fixed_zp,
                                         codes + row * cr, scales + row * sr, zps + row * zr);
          if (rc != ORC_OK) return rc;
        }
  return ORC_OK;
}

/*
 * INT4 decode attention. History rows come from the codes; when cur_kv
 * ([2, B, Hkv, 1, D] bf16) is given, the last visible token (position
 * lens[b] - 1, the one being appended) takes part uncompressed from cur_kv,
 * as the current K/V do before they are encoded.
 */
int orc_int4_attention(const uint16_t* q, int Hq, const uint8_t* codes, const uint16_t* scales,
                       const uint8_t* zps, int B, int Hkv, int C, int D, const int32_t* lens,
                       const uint16_t* cur_kv, double scale, int window, double* out) {
  if (B < 0 || Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0 || D <= 0 || D % 32 != 0) return ORC_ERR_SHAPE;
  for (int b = 0; b < B; ++b)
    if (lens[b] < 0 || lens[b] > C) return ORC_ERR_CAPACITY;
  int G = Hq / Hkv;
  int cr = codes_row(D), sr = scales_row(D), zr = zps_row(D);
  double* K = (double*)malloc(((size_t)C + 1) * D * sizeof(double));
  double* V = (double*)malloc(((size_t)C + 1) * D * sizeof(double));
  if (!K || !V) {
    free(K);
    free(V);
    return ORC_ERR_ALLOC;
  }
  int rc = ORC_OK;
  for (int b = 0; b < B && rc == ORC_OK; ++b) {
    int lo, hi;
    int n = orc_visible_range(lens[b], window, &lo, &hi);
    for (int g = 0; g < Hkv && rc == ORC_OK; ++g) {
      for (int t = 0; t < n; ++t) {
        int pos = lo + t;
        if (cur_kv && pos == hi - 1) {
          size_t kb = (((size_t)0 * B + b) * Hkv + g) * D;
          size_t vb = (((size_t)1 * B + b) * Hkv + g) * D;
          for (int d = 0; d < D; ++d) {
            K[(size_t)t * D + d] = bf16_to_double(cur_kv[kb + d]);
            V[(size_t)t * D + d] = bf16_to_double(cur_kv[vb + d]);
          }
          continue;
        }
        size_t krow = (((size_t)0 * B + b) * Hkv + g) * C + pos;
        size_t vrow = (((size_t)1 * B + b) * Hkv + g) * C + pos;
        orc_int4_dequantize_row(codes + krow * cr, scales + krow * sr, zps + krow * zr, D,
                                K + (size_t)t * D);
        orc_int4_dequantize_row(codes + vrow * cr, scales + vrow * sr, zps + vrow * zr, D,
                                V + (size_t)t * D);
      }
      rc = attend_group(q, ORC_BF16, Hq, G, b, g, D, K, V, n, scale, out);
    }
  }
  free(K);
  free(V);
  return rc;
}

/* ------------------------------------------- heterogeneous paged pages */

/*
 * A paged cache whose pages each carry their own K and V storage formats
 * (page "Persistent input/output feedback", sections Optional heterogeneous
 * paged KV and Selected-block quantization; the code packing of page "Custom,
 * quantized, and persistent values", affine branch: four-bit codes two per
 * byte and two-bit codes four per byte, least-significant bits first).
 *
 * Layout (the same one the library documents): num_pages slots of
 * 2 * Hkv * S * D * 4 bytes; plane k (0 = K, 1 = V) of page p starts at
 * p * slot + k * Hkv * S * D * 4; within a plane of format f the codes of
 * (head h, slot s) start at (h * S + s) * row_bytes(f) and hold the D
 * elements in order. Descriptor of a plane: format, scale, zero point.
 *
 * Formats: dense FLOAT, FLOAT16, BFLOAT16; affine INT8, UINT8, INT4, UINT4,
 * INT2, UINT2 with value = (code - zero_point) * scale.
 *   encode (QuantizeLinear): code = saturate(round_half_even(x / scale) + zp)
 *     to the type's range, in IEEE fp32; dense: the value rounded to nearest
 *     even in the dense type.
 *   decode (DequantizeLinear): (code - zp) * scale in fp32; dense: exact.
 */
enum { ORC_HF_F32 = 0, ORC_HF_F16, ORC_HF_BF16, ORC_HF_I8, ORC_HF_U8, ORC_HF_I4, ORC_HF_U4, ORC_HF_I2, ORC_HF_U2 };

typedef struct {
  int32_t format;
  float scale;
  int32_t zero_point;
} orc_plane_fmt;

typedef struct {
  orc_plane_fmt k, v;
} orc_page_desc;

int orc_hf_bits(int f) {
  switch (f) {
    case ORC_HF_F32: return 32;
    case ORC_HF_F16: case ORC_HF_BF16: return 16;
    case ORC_HF_I8: case ORC_HF_U8: return 8;
    case ORC_HF_I4: case ORC_HF_U4: return 4;
    case ORC_HF_I2: case ORC_HF_U2: return 2;
  }
  return 0;
}
static int hf_affine(int f) { return f >= ORC_HF_I8 && f <= ORC_HF_U2; }
static int hf_signed(int f) { return f == ORC_HF_I8 || f == ORC_HF_I4 || f == ORC_HF_I2; }
/* code range of an affine format */
void orc_hf_range(int f, int* qmin, int* qmax) {
  int bits = orc_hf_bits(f);
  if (hf_signed(f)) {
    *qmin = -(1 << (bits - 1));
    *qmax = (1 << (bits - 1)) - 1;
  } else {
    *qmin = 0;
    *qmax = (1 << bits) - 1;
  }
}
long long orc_hf_row_bytes(int f, int D) { return ((long long)D * orc_hf_bits(f) + 7) / 8; }

static uint16_t float_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40); /* quiet NaN */
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Encode one row of D bf16 values into `row` (row_bytes(format) bytes). */
static void hf_encode_row(const uint16_t* x, int D, const orc_plane_fmt* pf, uint8_t* row) {
  const int f = pf->format;
  memset(row, 0, (size_t)orc_hf_row_bytes(f, D));
  for (int d = 0; d < D; ++d) {
    float v = bf16_to_float(x[d]);
    if (f == ORC_HF_F32) {
      memcpy(row + 4 * (size_t)d, &v, 4);
    } else if (f == ORC_HF_F16) {
      uint16_t h = float_to_fp16_bits(v);
      memcpy(row + 2 * (size_t)d, &h, 2);
    } else if (f == ORC_HF_BF16) {
      uint16_t h = float_to_bf16_rne(v);
      memcpy(row + 2 * (size_t)d, &h, 2);
    } else {
      int qmin, qmax;
      orc_hf_range(f, &qmin, &qmax);
      float r = rintf(v / pf->scale) + (float)pf->zero_point;
      if (r < (float)qmin) r = (float)qmin;
      if (r > (float)qmax) r = (float)qmax;
      int code = (int)r;
      int bits = orc_hf_bits(f);
      unsigned u = (unsigned)code & ((1u << bits) - 1u); /* two's complement in `bits` */
      if (bits == 8)
        row[d] = (uint8_t)u;
      else
        row[(size_t)d * bits / 8] |= (uint8_t)(u << ((d * bits) % 8));
    }
  }
}

/* Decode one row into fp64 (each element is the fp32 reconstruction). */
static void hf_decode_row(const uint8_t* row, int D, const orc_plane_fmt* pf, double* out) {
  const int f = pf->format;
  for (int d = 0; d < D; ++d) {
    if (f == ORC_HF_F32) {
      float v;
      memcpy(&v, row + 4 * (size_t)d, 4);
      out[d] = v;
    } else if (f == ORC_HF_F16) {
      uint16_t h;
      memcpy(&h, row + 2 * (size_t)d, 2);
      out[d] = fp16_bits_to_double(h);
    } else if (f == ORC_HF_BF16) {
      uint16_t h;
      memcpy(&h, row + 2 * (size_t)d, 2);
      out[d] = bf16_to_double(h);
    } else {
      int bits = orc_hf_bits(f);
      unsigned u = bits == 8 ? row[d] : (row[(size_t)d * bits / 8] >> ((d * bits) % 8)) & ((1u << bits) - 1u);
      int code = (int)u;
      if (hf_signed(f) && code >= (1 << (bits - 1))) code -= (1 << bits);
      float v = (float)(code - pf->zero_point) * pf->scale;
      out[d] = v;
    }
  }
}

static int hf_check_fmt(const orc_plane_fmt* pf) {
  if (pf->format < ORC_HF_F32 || pf->format > ORC_HF_U2) return ORC_ERR_SHAPE;
  if (hf_affine(pf->format)) {
    int qmin, qmax;
    orc_hf_range(pf->format, &qmin, &qmax);
    if (!(pf->scale > 0.0f) || !isfinite(pf->scale)) return ORC_ERR_SHAPE;
    if (pf->zero_point < qmin || pf->zero_point > qmax) return ORC_ERR_SHAPE;
  }
  return ORC_OK;
}

int orc_hf_encode_row(const uint16_t* x, int D, const orc_plane_fmt* pf, uint8_t* row) {
  int rc = hf_check_fmt(pf);
  if (rc != ORC_OK) return rc;
  hf_encode_row(x, D, pf, row);
  return ORC_OK;
}
int orc_hf_decode_row(const uint8_t* row, int D, const orc_plane_fmt* pf, double* out) {
  int rc = hf_check_fmt(pf);
  if (rc != ORC_OK) return rc;
  hf_decode_row(row, D, pf, out);
  return ORC_OK;
}

static uint8_t* hf_row_ptr(uint8_t* pool, int Hkv, int S, int D, int page, int plane, int h, int s, int f) {
  size_t plane_bytes = (size_t)Hkv * S * D * 4;
  return pool + (size_t)page * 2 * plane_bytes + (size_t)plane * plane_bytes +
         ((size_t)h * S + s) * (size_t)orc_hf_row_bytes(f, D);
}

/*
 * Append new_len tokens per row at positions[b] (values [2, B, Hkv, new_len, D]
 * bf16). A token that lands in slot 0 of its page starts the page: the page
 * takes the formats `new_fmt` (K, V). Any other token is encoded in its page's
 * existing formats. Rejects bad positions, pages or formats before writing.
 */
int orc_hpaged_append(uint8_t* pool, orc_page_desc* desc, int P, int Hkv, int S, int D,
                      const int32_t* block_table, int M, int B, const uint16_t* values, int new_len,
                      const int32_t* positions, const orc_page_desc* new_fmt) {
  if (B < 0 || Hkv <= 0 || D <= 0 || S <= 0 || M < 0 || new_len < 0 || D % 4) return ORC_ERR_SHAPE;
  if (hf_check_fmt(&new_fmt->k) || hf_check_fmt(&new_fmt->v)) return ORC_ERR_SHAPE;
  for (int b = 0; b < B; ++b) {
    if (positions[b] < 0 || (long long)positions[b] + new_len > (long long)M * S) return ORC_ERR_CAPACITY;
    for (int j = 0; j < new_len; ++j) {
      int t = positions[b] + j;
      int page = block_table[(size_t)b * M + t / S];
      if (page < 0 || page >= P) return ORC_ERR_PAGE;
    }
  }
  for (int b = 0; b < B; ++b)
    for (int j = 0; j < new_len; ++j) {
      int t = positions[b] + j;
      int page = block_table[(size_t)b * M + t / S];
      int s = t % S;
      if (s == 0) desc[page] = *new_fmt;
      for (int plane = 0; plane < 2; ++plane) {
        const orc_plane_fmt* pf = plane == 0 ? &desc[page].k : &desc[page].v;
        for (int h = 0; h < Hkv; ++h) {
          const uint16_t* x = values + ((((size_t)plane * B + b) * Hkv + h) * new_len + j) * D;
          hf_encode_row(x, D, pf, hf_row_ptr(pool, Hkv, S, D, page, plane, h, s, pf->format));
        }
      }
    }
  return ORC_OK;
}

/*
 * Decode attention over the heterogeneous pages: the visible tokens of row b
 * decoded by their pages' formats; with cur_kv ([2, B, Hkv, 1, D] bf16) the
 * token at lens[b] - 1 takes part uncompressed from cur_kv (the current K/V
 * are attended before they are encoded). q [B, Hq, D] bf16; out fp64.
 */
int orc_hpaged_attention(const uint16_t* q, int Hq, const uint8_t* pool, const orc_page_desc* desc, int P,
                         int Hkv, int S, int D, const int32_t* block_table, int M, int B, const int32_t* lens,
                         const uint16_t* cur_kv, double scale, int window, double* out) {
  if (B < 0 || Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0 || D <= 0 || S <= 0 || M < 0 || D % 4) return ORC_ERR_SHAPE;
  long long cap = (long long)M * S;
  for (int b = 0; b < B; ++b) {
    if (lens[b] < 0 || lens[b] > cap) return ORC_ERR_CAPACITY;
    for (int t = 0; t < lens[b]; ++t) {
      int page = block_table[(size_t)b * M + t / S];
      if (page < 0 || page >= P) return ORC_ERR_PAGE;
      if (hf_check_fmt(&desc[page].k) || hf_check_fmt(&desc[page].v)) return ORC_ERR_SHAPE;
    }
  }
  int G = Hq / Hkv;
  double* K = (double*)malloc(((size_t)cap + 1) * D * sizeof(double));
  double* V = (double*)malloc(((size_t)cap + 1) * D * sizeof(double));
  if (!K || !V) {
    free(K);
    free(V);
    return ORC_ERR_ALLOC;
  }
  int rc = ORC_OK;
  for (int b = 0; b < B && rc == ORC_OK; ++b) {
    int lo, hi;
    int n = orc_visible_range(lens[b], window, &lo, &hi);
    for (int g = 0; g < Hkv && rc == ORC_OK; ++g) {
      for (int t = 0; t < n; ++t) {
        int logical = lo + t;
        if (cur_kv && logical == lens[b] - 1) {
          for (int d = 0; d < D; ++d) {
            K[(size_t)t * D + d] = bf16_to_double(cur_kv[(((size_t)0 * B + b) * Hkv + g) * D + d]);
            V[(size_t)t * D + d] = bf16_to_double(cur_kv[(((size_t)1 * B + b) * Hkv + g) * D + d]);
          }
          continue;
        }
        int page = block_table[(size_t)b * M + logical / S];
        int s = logical % S;
        hf_decode_row(hf_row_ptr((uint8_t*)pool, Hkv, S, D, page, 0, g, s, desc[page].k.format), D,
                      &desc[page].k, K + (size_t)t * D);
        hf_decode_row(hf_row_ptr((uint8_t*)pool, Hkv, S, D, page, 1, g, s, desc[page].v.format), D,
                      &desc[page].v, V + (size_t)t * D);
      }
      rc = attend_group(q, ORC_BF16, Hq, G, b, g, D, K, V, n, scale, out);
    }
  }
  free(K);
  free(V);
  return rc;
}

/*
 * QuantizePagedCache on the selected pages (unique indices): each page's valid
 * prefix of valid[i] slots is decoded in its current formats and encoded in
 * `to` (K, V independently); the other slots become the destination format's
 * zeros (encode of 0). Every index, length and format is checked before any
 * page changes.
 */
int orc_hpaged_quantize(uint8_t* pool, orc_page_desc* desc, int P, int Hkv, int S, int D, const int32_t* pages,
                        const int32_t* valid, int n, const orc_page_desc* to) {
  if (Hkv <= 0 || D <= 0 || S <= 0 || n < 0 || D % 4) return ORC_ERR_SHAPE;
  if (hf_check_fmt(&to->k) || hf_check_fmt(&to->v)) return ORC_ERR_SHAPE;
  for (int i = 0; i < n; ++i) {
    if (pages[i] < 0 || pages[i] >= P) return ORC_ERR_PAGE;
    if (valid[i] < 0 || valid[i] > S) return ORC_ERR_CAPACITY;
    for (int j = 0; j < i; ++j)
      if (pages[j] == pages[i]) return ORC_ERR_SHAPE;
  }
  double* vals = (double*)malloc((size_t)Hkv * S * D * sizeof(double));
  float* x = (float*)malloc((size_t)D * sizeof(float));
  if (!vals || !x) {
    free(vals);
    free(x);
    return ORC_ERR_ALLOC;
  }
  for (int i = 0; i < n; ++i) {
    int page = pages[i];
    for (int plane = 0; plane < 2; ++plane) {
      orc_plane_fmt* from = plane == 0 ? &desc[page].k : &desc[page].v;
      const orc_plane_fmt* dst = plane == 0 ? &to->k : &to->v;
      /* the whole plane is decoded before any of it is rewritten: source and
         destination rows share the page's bytes */
      for (int h = 0; h < Hkv; ++h)
        for (int s = 0; s < valid[i]; ++s)
          hf_decode_row(hf_row_ptr(pool, Hkv, S, D, page, plane, h, s, from->format), D, from,
                        vals + ((size_t)h * S + s) * D);
      for (int h = 0; h < Hkv; ++h)
        for (int s = 0; s < S; ++s) {
          uint8_t* row = hf_row_ptr(pool, Hkv, S, D, page, plane, h, s, dst->format);
          for (int d = 0; d < D; ++d) x[d] = s < valid[i] ? (float)vals[((size_t)h * S + s) * D + d] : 0.0f;
          /* encode from the fp32 reconstruction (a float, not rounded to bf16 first) */
          if (dst->format == ORC_HF_F32) {
            memcpy(row, x, (size_t)D * 4);
          } else if (dst->format == ORC_HF_F16 || dst->format == ORC_HF_BF16) {
            for (int d = 0; d < D; ++d) {
              uint16_t hb = dst->format == ORC_HF_F16 ? float_to_fp16_bits(x[d]) : float_to_bf16_rne(x[d]);
              memcpy(row + 2 * (size_t)d, &hb, 2);
            }
          } else {
            int qmin, qmax, bits = orc_hf_bits(dst->format);
            orc_hf_range(dst->format, &qmin, &qmax);
            memset(row, 0, (size_t)orc_hf_row_bytes(dst->format, D));
            for (int d = 0; d < D; ++d) {
              float r = rintf(x[d] / dst->scale) + (float)dst->zero_point;
              if (r < (float)qmin) r = (float)qmin;
              if (r > (float)qmax) r = (float)qmax;
              unsigned u = (unsigned)(int)r & ((1u << bits) - 1u);
              if (bits == 8)
                row[d] = (uint8_t)u;
              else
                row[(size_t)d * bits / 8] |= (uint8_t)(u << ((d * bits) % 8));
            }
          }
        }
      *from = *dst;
    }
  }
  free(vals);
  free(x);
  return ORC_OK;
}
