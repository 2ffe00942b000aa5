/*
 * mxg_oracle.c -- plain, slow, obviously-correct CPU reference for the grouped
 * block-scaled quantize + grouped GEMM path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file.  Only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA implementation.
 *
 * Sources (the three web pages this method is described on):
 *   [TE-gemm]  TransformerEngine transformer_engine/jax/cpp_extensions/gemm.py
 *              (commit 070b5b7): swizzled_scale, _get_nvfp4_tensor_scale_inv,
 *              _jax_scaled_matmul, grouped_gemm.
 *   [PR2763]   TransformerEngine PR #2763 "[JAX] MXFP8 Grouped Quant+GEMM":
 *              description, the offsets-kernel review thread and the
 *              workspace-layout review thread.
 *   [PR3661]   TransformerEngine PR #3661 "Add row-scaled NVFP4 support to
 *              grouped-tensor GEMM": description and commit messages.
 *
 * Where the pages leave a rule open the reading taken is stated at the
 * function (MXFP8 scale rule "R1", NVFP4 row-scaled rule "R2", nibble order,
 * offsets sanitisation).  Floating-point decisions that pick an integer code
 * are made in fp64 where the scaled value is exact (MXFP8) and in IEEE fp32
 * round-to-nearest, one operation at a time, where the rule itself is stated
 * in fp32 (NVFP4 R2).  Build with -ffp-contract=off so no multiply-add is
 * fused.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* Status bits shared by meaning (not by code) with the device status word. */
#define ORACLE_ST_NEG_SIZE 1
#define ORACLE_ST_MISALIGNED 2
#define ORACLE_ST_SUM_OVER_CAPACITY 4

/* ------------------------------------------------------------------------ */
/* Element formats (OCP Microscaling v1.0 definitions; NVFP4 usage in        */
/* [TE-gemm] _get_nvfp4_tensor_scale_inv: data max 6 (E2M1), scale max 448). */
/* ------------------------------------------------------------------------ */

/* bf16 bit pattern -> fp32 (exact: bf16 is the top half of an fp32). */
static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* E4M3 (fn variant): s.eeee.mmm, bias 7, no infinities, 0x7F/0xFF = NaN. */
ORACLE_API double mxg_oracle_e4m3_decode(uint8_t b) {
  int s = b >> 7, e = (b >> 3) & 0xF, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9); /* subnormal: m * 2^-9 */
  else
    v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/* Round-to-nearest-even onto the E4M3 grid, saturating finite values to
 * +-448 ("satfinite").  In every binade the grid step is q = 2^(e-3) with
 * e = max(floor(log2|v|), -6); rint() rounds half to even, and the even
 * multiple of q is the code with an even mantissa. */
ORACLE_API uint8_t mxg_oracle_e4m3_encode(double v) {
  uint8_t s = signbit(v) ? 0x80 : 0x00;
  double a = fabs(v), q, n, r;
  int E, e;
  if (isnan(v)) return 0x7F;
  if (a >= 448.0) return s | 0x7E;
  if (a == 0.0) return s;
  frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) */
  e = E - 1;
  if (e < -6) e = -6;
  q = ldexp(1.0, e - 3);
  n = rint(a / q);
  r = n * q;
  if (r == 0.0) return s;
  if (r < ldexp(1.0, -6)) return s | (uint8_t)n; /* subnormal: code = r / 2^-9 */
  frexp(r, &E);
  e = E - 1;
  {
    int mant = (int)(r / ldexp(1.0, e - 3)) - 8;
    return s | (uint8_t)(((e + 7) << 3) | mant);
  }
}

/* E2M1: s.ee.m, bias 1; magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}. */
ORACLE_API double mxg_oracle_e2m1_decode(uint8_t nib) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  double v = mag[nib & 7];
  return (nib & 8) ? -v : v;
}

/* Round-to-nearest-even onto the E2M1 grid, saturating to +-6. */
ORACLE_API uint8_t mxg_oracle_e2m1_encode(double v) {
  uint8_t s = signbit(v) ? 0x8 : 0x0;
  double a = fabs(v), q, r;
  if (isnan(v)) return 0x7; /* unpinned: configs are finite */
  if (a >= 6.0) return s | 0x7;
  q = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
  r = rint(a / q) * q;
  if (r == 0.0) return s;
  if (r == 0.5) return s | 1;
  if (r == 1.0) return s | 2;
  if (r == 1.5) return s | 3;
  if (r == 2.0) return s | 4;
  if (r == 3.0) return s | 5;
  if (r == 4.0) return s | 6;
  return s | 7; /* 6.0 */
}

/* E8M0: byte b is 2^(b-127); 0xFF is NaN. */
ORACLE_API double mxg_oracle_e8m0_decode(uint8_t b) {
  if (b == 0xFF) return NAN;
  return ldexp(1.0, (int)b - 127);
}

/* ------------------------------------------------------------------------ */
/* R1: the MXFP8 block scale.  The pages fix the format (one E8M0 scale per  */
/* 1x32 block, [TE-gemm] _jax_scaled_matmul / scaling modes) but not the    */
/* rule.  Reading taken: the smallest power of two 2^e with                  */
/* amax <= 448 * 2^e, i.e. e = ceil(log2(amax / 448)), clamped to           */
/* [-127, 127]; an all-zero block gets e = -127 (byte 0x00).                */
/* With amax = m * 2^E, m in [1, 2): e = E - 8 + (m > 1.75).                 */
/* ------------------------------------------------------------------------ */
ORACLE_API int mxg_oracle_mx_scale_exponent(float amax) {
  int E, e;
  double f;
  if (!(amax > 0.0f)) return -127;
  f = frexp((double)amax, &E); /* amax = (2f) * 2^(E-1), 2f in [1, 2) */
  e = (E - 1) - 8 + ((2.0 * f > 1.75) ? 1 : 0);
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

/* ------------------------------------------------------------------------ */
/* Scale-factor swizzle, [TE-gemm] swizzled_scale: S[R, C] is reshaped to   */
/* (R/128, 4, 32, C/4, 4), the axes are permuted to (0, 3, 2, 1, 4) and the */
/* result is flattened.  Written out as a flat index.  Requires R % 128 == 0 */
/* and C % 4 == 0.                                                           */
/* ------------------------------------------------------------------------ */
ORACLE_API int64_t mxg_oracle_swizzle_index(int64_t r, int64_t c, int64_t C) {
  int64_t r0 = r / 128, r1 = (r % 128) / 32, r2 = r % 32;
  int64_t c0 = c / 4, c1 = c % 4;
  return (((r0 * (C / 4) + c0) * 32 + r2) * 4 + r1) * 4 + c1;
}

/* Inverse of the swizzle: unswizzled[r*C + c] = swizzled[index(r, c)]
 * ([PR2763] _unswizzle_mxfp8_grouped_scale used by the dequantizer). */
ORACLE_API void mxg_oracle_unswizzle(const uint8_t* swz, int64_t R, int64_t C, uint8_t* plain) {
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < C; ++c) plain[r * C + c] = swz[mxg_oracle_swizzle_index(r, c, C)];
}

ORACLE_API void mxg_oracle_swizzle(const uint8_t* plain, int64_t R, int64_t C, uint8_t* swz) {
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < C; ++c) swz[mxg_oracle_swizzle_index(r, c, C)] = plain[r * C + c];
}

/* ------------------------------------------------------------------------ */
/* Group sizes -> int64 sizes and element offsets.                          */
/* [PR2763] description: int32 group sizes are widened to int64 and scaled  */
/* by a multiplier; offsets review thread: offsets[0] = 0,                  */
/* offsets[i] = sum_{j<i} first_dims[j] * last_dim, G+1 values; workspace   */
/* review thread: [G int64 sizes | G+1 int64 offsets].                      */
/* Reading taken for the multiplier: rows per size unit.                    */
/* Sanitisation (not on the pages; this library's contract): a negative    */
/* size counts as 0 (NEG_SIZE), a size that is not a multiple of 128 rows   */
/* is rounded down to one (MISALIGNED), and rows beyond rows_capacity are   */
/* cut off (SUM_OVER_CAPACITY).  The workspace holds the sanitised sizes.   */
/* Returns the status bits.                                                 */
/* ------------------------------------------------------------------------ */
static int32_t group_offsets_rule(const int64_t* sizes, int G, int64_t multiplier,
                                  int64_t last_dim, int64_t rows_capacity, int64_t* ws,
                                  int round128) {
  int32_t st = 0;
  int64_t rows_before = 0;
  ws[G] = 0;
  for (int g = 0; g < G; ++g) {
    int64_t s = sizes[g] * multiplier;
    if (s < 0) {
      st |= ORACLE_ST_NEG_SIZE;
      s = 0;
    }
    if (round128 && s % 128 != 0) {
      st |= ORACLE_ST_MISALIGNED;
      s -= s % 128;
    }
    if (s > rows_capacity - rows_before) {
      st |= ORACLE_ST_SUM_OVER_CAPACITY;
      s = rows_capacity - rows_before;
    }
    ws[g] = s;
    rows_before += s;
    ws[G + 1 + g] = ws[G + g] + s * last_dim;
  }
  return st;
}

/* Sizes rounded down to multiples of 128 (the aligned contract). */
ORACLE_API int32_t mxg_oracle_group_offsets(const int64_t* sizes, int G, int64_t multiplier,
                                            int64_t last_dim, int64_t rows_capacity, int64_t* ws) {
  return group_offsets_rule(sizes, G, multiplier, last_dim, rows_capacity, ws, 1);
}

/* Sizes kept as given (groups of any size: [PR2763] review thread, the
   128-row rule comes from the offset arithmetic of the quantize and GEMM
   setup, not from the GEMM). */
ORACLE_API int32_t mxg_oracle_group_offsets_unaligned(const int64_t* sizes, int G,
                                                      int64_t multiplier, int64_t last_dim,
                                                      int64_t rows_capacity, int64_t* ws) {
  return group_offsets_rule(sizes, G, multiplier, last_dim, rows_capacity, ws, 0);
}

/* ------------------------------------------------------------------------ */
/* MXFP8 grouped quantize.  Groups are 128-row aligned, so the per-group    */
/* quantize over rows [0, rows_live) equals the dense quantize of those     */
/* rows and group g's scales start at byte off_g * cols / 32 of the global  */
/* swizzled layout ([PR2763], GEMM-setup review thread: scale pointer =     */
/* data offset / 32).  Rows >= rows_live are neither read nor written.      */
/* ------------------------------------------------------------------------ */

/* Rowwise: 1x32 blocks along cols.  q[rows_cap, cols] E4M3,
 * sf = swizzled [rows_cap, cols/32] E8M0. */
ORACLE_API void mxg_oracle_mxfp8_quantize_rowwise(const uint16_t* x, int64_t rows_live,
                                                  int64_t cols, uint8_t* q, uint8_t* sf) {
  const int64_t C = cols / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows_live; ++r) {
    for (int64_t b = 0; b < C; ++b) {
      const uint16_t* xb = x + r * cols + b * 32;
      float amax = 0.0f;
      int e;
      for (int i = 0; i < 32; ++i) {
        float a = fabsf(bf16_to_f32(xb[i]));
        if (a > amax) amax = a;
      }
      e = mxg_oracle_mx_scale_exponent(amax);
      sf[mxg_oracle_swizzle_index(r, b, C)] = (uint8_t)(e + 127);
      for (int i = 0; i < 32; ++i)
        q[r * cols + b * 32 + i] = mxg_oracle_e4m3_encode(ldexp((double)bf16_to_f32(xb[i]), -e));
    }
  }
}

/* Colwise, written transposed ([TE-gemm] swizzled_scale, is_colwise branch:
 * the colwise scale matrix is transposed before the swizzle).  32x1 blocks
 * along rows.  qT[cols, rows_cap] E4M3 holds qT[k, m] = Q(x[m, k]);
 * sfT = swizzled [cols, rows_cap/32] E8M0.  rows_live % 32 == 0. */
ORACLE_API void mxg_oracle_mxfp8_quantize_colwise(const uint16_t* x, int64_t rows_live,
                                                  int64_t rows_cap, int64_t cols, uint8_t* qT,
                                                  uint8_t* sfT) {
  const int64_t C = rows_cap / 32;
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < cols; ++k) {
    for (int64_t j = 0; j < rows_live / 32; ++j) {
      float amax = 0.0f;
      int e;
      for (int i = 0; i < 32; ++i) {
        float a = fabsf(bf16_to_f32(x[(j * 32 + i) * cols + k]));
        if (a > amax) amax = a;
      }
      e = mxg_oracle_mx_scale_exponent(amax);
      sfT[mxg_oracle_swizzle_index(k, j, C)] = (uint8_t)(e + 127);
      for (int i = 0; i < 32; ++i)
        qT[k * rows_cap + j * 32 + i] =
            mxg_oracle_e4m3_encode(ldexp((double)bf16_to_f32(x[(j * 32 + i) * cols + k]), -e));
    }
  }
}

/* ------------------------------------------------------------------------ */
/* R2: row-scaled NVFP4 quantize.  The pages give the outer scale as        */
/* amax / (E2M1 max * E4M3 max) = amax / 2688 ([TE-gemm]                    */
/* _get_nvfp4_tensor_scale_inv), applied per row ([PR3661] description:     */
/* per-row FP32 outer scale), with E2M1 data and E4M3 scales per 1x16       */
/* block.  Reading taken for the block rule, every step an IEEE fp32        */
/* round-to-nearest operation in this order:                                */
/*   A   = max_k |x[r,k]|,  s_r = A / 2688          (stored outer scale)    */
/*   S   = 2688 / A                                                         */
/*   per 16-block: t = (amax_b / 6) * S,  sb = E4M3_RNE_satfinite(t)        */
/*   if sb == 0 the block's codes are signed zeros, else                    */
/*   v = x * (S / sb),  code = E2M1_RNE_satfinite(v)                        */
/* A == 0 gives s_r = 0, zero scale bytes and signed-zero codes.            */
/* Packing: element 2i in the low nibble of byte i, 2i+1 in the high one.   */
/* q[rows, cols/2], sf = swizzled [rows_cap, cols/16] E4M3, outer[rows].    */
/* ------------------------------------------------------------------------ */
ORACLE_API void mxg_oracle_nvfp4_quantize_rowwise(const uint16_t* x, int64_t rows_live,
                                                  int64_t cols, uint8_t* q, uint8_t* sf,
                                                  float* outer) {
  const int64_t C = cols / 16;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows_live; ++r) {
    const uint16_t* xr = x + r * cols;
    float A = 0.0f, S, t, sbv, ratio, v;
    for (int64_t k = 0; k < cols; ++k) {
      float a = fabsf(bf16_to_f32(xr[k]));
      if (a > A) A = a;
    }
    if (A == 0.0f) {
      outer[r] = 0.0f;
      for (int64_t b = 0; b < C; ++b) sf[mxg_oracle_swizzle_index(r, b, C)] = 0;
      for (int64_t k = 0; k < cols; k += 2) {
        uint8_t lo = signbit(bf16_to_f32(xr[k])) ? 0x8 : 0x0;
        uint8_t hi = signbit(bf16_to_f32(xr[k + 1])) ? 0x8 : 0x0;
        q[r * (cols / 2) + k / 2] = (uint8_t)(lo | (hi << 4));
      }
      continue;
    }
    outer[r] = A / 2688.0f;
    S = 2688.0f / A;
    for (int64_t b = 0; b < C; ++b) {
      float ab = 0.0f;
      uint8_t sbyte, codes[16];
      for (int i = 0; i < 16; ++i) {
        float a = fabsf(bf16_to_f32(xr[b * 16 + i]));
        if (a > ab) ab = a;
      }
      t = ab / 6.0f;
      t = t * S;
      sbyte = mxg_oracle_e4m3_encode((double)t) & 0x7F;
      sf[mxg_oracle_swizzle_index(r, b, C)] = sbyte;
      sbv = (float)mxg_oracle_e4m3_decode(sbyte);
      for (int i = 0; i < 16; ++i) {
        float xv = bf16_to_f32(xr[b * 16 + i]);
        if (sbv == 0.0f) {
          codes[i] = signbit(xv) ? 0x8 : 0x0;
        } else {
          ratio = S / sbv;
          v = xv * ratio;
          codes[i] = mxg_oracle_e2m1_encode((double)v);
        }
      }
      for (int i = 0; i < 16; i += 2)
        q[r * (cols / 2) + (b * 16 + i) / 2] = (uint8_t)(codes[i] | (codes[i + 1] << 4));
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Dequantize ([PR2763] dequantizer: unswizzle the scales, then decode      */
/* data * scale).  Rows are given as an index list so callers can sample.   */
/* out[i*cols + k] = value of row row_idx[i], column k, in fp64.            */
/* ------------------------------------------------------------------------ */
ORACLE_API void mxg_oracle_mxfp8_dequantize_rows(const uint8_t* q, const uint8_t* sf, int64_t cols,
                                                 const int64_t* row_idx, int64_t n_rows,
                                                 double* out) {
  const int64_t C = cols / 32;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t r = row_idx[i];
    for (int64_t k = 0; k < cols; ++k) {
      double s = mxg_oracle_e8m0_decode(sf[mxg_oracle_swizzle_index(r, k / 32, C)]);
      out[i * cols + k] = mxg_oracle_e4m3_decode(q[r * cols + k]) * s;
    }
  }
}

/* NVFP4: value = e2m1(code) * e4m3(block scale) * outer[r].  When
 * with_outer == 0 the outer scale is left out (the "neutral outer scale"
 * operand of [PR3661]). */
ORACLE_API void mxg_oracle_nvfp4_dequantize_rows(const uint8_t* q, const uint8_t* sf,
                                                 const float* outer, int with_outer, int64_t cols,
                                                 const int64_t* row_idx, int64_t n_rows,
                                                 double* out) {
  const int64_t C = cols / 16;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t r = row_idx[i];
    double o = with_outer ? (double)outer[r] : 1.0;
    for (int64_t k = 0; k < cols; ++k) {
      uint8_t byte = q[r * (cols / 2) + k / 2];
      uint8_t nib = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      double s = mxg_oracle_e4m3_decode(sf[mxg_oracle_swizzle_index(r, k / 16, C)]);
      out[i * cols + k] = mxg_oracle_e2m1_decode(nib) * s * o;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Array forms of the codecs and of R1, used by the pin tests.              */
/* ------------------------------------------------------------------------ */
ORACLE_API void mxg_oracle_e4m3_encode_array(const double* v, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = mxg_oracle_e4m3_encode(v[i]);
}

ORACLE_API void mxg_oracle_e2m1_encode_array(const double* v, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = mxg_oracle_e2m1_encode(v[i]);
}

ORACLE_API void mxg_oracle_mx_scale_exponent_array(const float* amax, int64_t n, int32_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = mxg_oracle_mx_scale_exponent(amax[i]);
}

/* ------------------------------------------------------------------------ */
/* R2 applied colwise, written transposed: the columnwise copy PR #3661      */
/* enables for wgrad, with one amax per column and expert.                  */
/* Reading taken: for group g and column k the outer scale                  */
/* is s[g, k] = A / 2688 with A = max over the group's rows of |x[m, k]|;   */
/* then R2 runs along m over 16-row blocks (groups are 128-row aligned, so  */
/* blocks never straddle groups).  Output qT[k, m/2] packs rows m (low      */
/* nibble, even m) and m+1; scales swizzled over [cols, rows_cap/16];      */
/* outer [G, cols].  group_rows: int64 row offsets [G+1].                   */
/* ------------------------------------------------------------------------ */
ORACLE_API void mxg_oracle_nvfp4_quantize_colwise(const uint16_t* x, const int64_t* group_rows,
                                                  int G, int64_t rows_cap, int64_t cols,
                                                  uint8_t* qT, uint8_t* sfT, float* outer) {
  const int64_t C = rows_cap / 16;
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < cols; ++k) {
    for (int g = 0; g < G; ++g) {
      const int64_t lo = group_rows[g], hi = group_rows[g + 1];
      float A = 0.0f, S, t, sbv, ratio, v;
      if (hi <= lo) {
        outer[(int64_t)g * cols + k] = 0.0f;
        continue;
      }
      for (int64_t m = lo; m < hi; ++m) {
        float a = fabsf(bf16_to_f32(x[m * cols + k]));
        if (a > A) A = a;
      }
      outer[(int64_t)g * cols + k] = A == 0.0f ? 0.0f : A / 2688.0f;
      S = A == 0.0f ? 0.0f : 2688.0f / A;
      for (int64_t m0 = lo; m0 < hi; m0 += 16) {
        float ab = 0.0f;
        uint8_t sbyte = 0, codes[16];
        for (int i = 0; i < 16; ++i) {
          float a = fabsf(bf16_to_f32(x[(m0 + i) * cols + k]));
          if (a > ab) ab = a;
        }
        if (A != 0.0f) {
          t = ab / 6.0f;
          t = t * S;
          sbyte = mxg_oracle_e4m3_encode((double)t) & 0x7F;
        }
        sfT[mxg_oracle_swizzle_index(k, m0 / 16, C)] = sbyte;
        sbv = (float)mxg_oracle_e4m3_decode(sbyte);
        for (int i = 0; i < 16; ++i) {
          float xv = bf16_to_f32(x[(m0 + i) * cols + k]);
          if (sbv == 0.0f) {
            codes[i] = signbit(xv) ? 0x8 : 0x0;
          } else {
            ratio = S / sbv;
            v = xv * ratio;
            codes[i] = mxg_oracle_e2m1_encode((double)v);
          }
        }
        for (int i = 0; i < 16; i += 2)
          qT[k * (rows_cap / 2) + (m0 + i) / 2] = (uint8_t)(codes[i] | (codes[i + 1] << 4));
      }
    }
  }
}
