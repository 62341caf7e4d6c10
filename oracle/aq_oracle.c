/*
 * aq_oracle.c -- CPU oracle for the NVFP4 decode-projection path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE (see aq_oracle.h for who may use it
 * and for the list of sources [H] [R] [Q] [B] [P] [W] [F] cited below).
 *
 * Build: cc -std=c11 -O2 -fno-fast-math -ffp-contract=off -fPIC -shared.
 * The code relies on C float arithmetic being evaluated in binary32
 * (FLT_EVAL_METHOD == 0, true on x86-64 and aarch64) and on the default
 * round-to-nearest-even mode for rintf.
 */
#include "aq_oracle.h"

#include <float.h>
#include <math.h>
#include <string.h>

#if defined(FLT_EVAL_METHOD) && FLT_EVAL_METHOD != 0
#error "the oracle needs float expressions evaluated in binary32"
#endif

/* ------------------------------------------------------------------ bf16 */

float aqo_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round a binary32 to the nearest bf16, ties to the even significand: add
 * half of the dropped range, plus one if the kept lsb is odd, then truncate. */
uint16_t aqo_f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
  uint32_t keep_lsb = (u >> 16) & 1u;
  u += 0x7FFFu + keep_lsb;
  return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ E4M3 */

/* [F] float8_e4m3fn: sign, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 is subnormal (m * 2^-9); 0x7F / 0xFF are NaN; there is
 * no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448. */
float aqo_e4m3_decode(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  if (e == 15 && m == 7) return NAN;
  float mag = (e == 0) ? ldexpf((float)m, -9)          /* m/8 * 2^-6   */
                       : ldexpf((float)(8 + m), e - 10); /* (1+m/8)*2^(e-7) */
  return sign ? -mag : mag;
}

/* R4: round to nearest, ties to an even mantissa, saturate at 448. */
uint8_t aqo_e4m3_encode_satfinite(float t) {
  if (isnan(t)) return 0x7F;
  uint8_t sign = signbit(t) ? 0x80 : 0x00;
  float a = fabsf(t);
  if (a >= 448.0f) return (uint8_t)(sign | 0x7E);
  if (a < ldexpf(1.0f, -6)) {
    /* subnormal range: the grid step is 2^-9; scaling by 2^9 is exact, and
     * rintf rounds half to even.  A result of 8 is the code of 2^-6, the
     * smallest normal, because the code space is monotone. */
    int q = (int)rintf(ldexpf(a, 9));
    return (uint8_t)(sign | q);
  }
  int e2;
  frexpf(a, &e2);  /* a = f * 2^e2 with f in [0.5, 1) */
  int ue = e2 - 1; /* a in [2^ue, 2^(ue+1)), ue in [-6, 8] */
  int q = (int)rintf(ldexpf(a, 3 - ue)); /* significand * 8, in [8, 16] */
  if (q == 16) {
    q = 8;
    ue += 1;
  }
  /* a < 448 keeps ue <= 8 and, at ue == 8, q <= 14 (1.75 * 2^8). */
  return (uint8_t)(sign | ((ue + 7) << 3) | (q - 8));
}

/* ------------------------------------------------------------------ E2M1 */

/* [F] E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit.  Exponent field
 * 0 is subnormal (m * 0.5); the magnitudes are 0, .5, 1, 1.5, 2, 3, 4, 6. */
float aqo_e2m1_decode(uint8_t nibble) {
  int sign = (nibble >> 3) & 1;
  int e = (nibble >> 1) & 3;
  int m = nibble & 1;
  float mag = (e == 0) ? 0.5f * (float)m : ldexpf((float)(2 + m), e - 2);
  return sign ? -mag : mag;
}

/* R5: round to nearest with ties to an even mantissa (0.25->0, 0.75->1,
 * 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4), saturate at 6, and keep the sign
 * bit of v even when the magnitude rounds to zero. */
uint8_t aqo_e2m1_encode_satfinite(float v) {
  uint8_t sign = signbit(v) ? 0x8 : 0x0;
  float a = fabsf(v);
  if (isnan(v) || a >= 6.0f) return (uint8_t)(sign | 0x7);
  if (a < 1.0f) {
    /* subnormal range, step 0.5: q in {0, 1, 2}; 2 is the code of 1.0 */
    int q = (int)rintf(a * 2.0f);
    return (uint8_t)(sign | q);
  }
  int e2;
  frexpf(a, &e2);
  int ue = e2 - 1;                       /* 0, 1 or 2 */
  int q = (int)rintf(ldexpf(a, 1 - ue)); /* significand * 2, in [2, 4] */
  if (q == 4) {
    q = 2;
    ue += 1;
  }
  if (ue > 2) return (uint8_t)(sign | 0x7); /* cannot happen for a < 6 */
  return (uint8_t)(sign | ((ue + 1) << 1) | (q - 2));
}

/* ------------------------------------------------------------ reconstruct */

/* [H] W_eff = s*W0 + U*V^T, R1: the low-rank term is summed first in fp32
 * (fmaf, r ascending, from +0); when it is zero the result is the plain
 * product s*W0 (so s = 1, U = V = 0 returns W0 bit-for-bit, [P], including
 * -0); otherwise s*W0 + delta is one fmaf; the fp32 result is rounded once
 * to bf16. */
void aqo_reconstruct(const uint16_t *W0, const float *s, const uint16_t *U,
                     const uint16_t *V, int64_t n, int64_t k, int64_t r,
                     uint16_t *W_eff) {
  for (int64_t i = 0; i < n; ++i) {
    for (int64_t j = 0; j < k; ++j) {
      float delta = 0.0f;
      for (int64_t t = 0; t < r; ++t)
        delta = fmaf(aqo_bf16_to_f32(U[i * r + t]),
                     aqo_bf16_to_f32(V[j * r + t]), delta);
      float w0 = aqo_bf16_to_f32(W0[i * k + j]);
      float e = (delta == 0.0f) ? s[i] * w0 : fmaf(s[i], w0, delta);
      W_eff[i * k + j] = aqo_f32_to_bf16_rne(e);
    }
  }
}

/* ------------------------------------------------------ per-tensor scale */

float aqo_amax_bf16(const uint16_t *W, int64_t count) {
  float a = 0.0f;
  for (int64_t i = 0; i < count; ++i) {
    float v = fabsf(aqo_bf16_to_f32(W[i]));
    if (isnan(v)) return NAN;
    if (v > a) a = v;
  }
  return a;
}

/* R2: 2688 = 6 (largest E2M1) * 448 (largest E4M3): the block holding the
 * tensor's largest magnitude gets the top E4M3 scale and its largest
 * element the top E2M1 code. */
int aqo_global_scales(float amax, float *g_enc, float *g_dec) {
  if (!isfinite(amax) || amax < 0.0f) return AQO_ERR_RANGE;
  if (amax == 0.0f) {
    *g_enc = 1.0f;
    *g_dec = 1.0f;
    return AQO_OK;
  }
  float ge = 2688.0f / amax;
  if (!isfinite(ge)) return AQO_ERR_RANGE;
  *g_enc = ge;
  *g_dec = amax / 2688.0f;
  return AQO_OK;
}

/* --------------------------------------------------------------- quantise */

/* [Q][R][F] One 16-element block along k (R3):
 *   b  = max |w| over the block
 *   t  = (b / 6) * g_enc              two fp32 operations
 *   sf = E4M3(t), sd = decode(sf)     round-to-nearest-even, satfinite
 *   sd == 0: every nibble of the block is 0                          (R4)
 *   else r = g_enc / sd (one division per block), q = E2M1(w * r)    (R5)
 * R6: byte i of a row holds element 2i in its low nibble, 2i+1 high. */
void aqo_quantize_rows(const uint16_t *W, int64_t rows, int64_t k, float g_enc,
                       uint8_t *packed, uint8_t *scales) {
  const int64_t nblk = k / 16;
  for (int64_t i = 0; i < rows; ++i) {
    for (int64_t j = 0; j < nblk; ++j) {
      const uint16_t *blk = W + i * k + j * 16;
      float b = 0.0f;
      for (int e = 0; e < 16; ++e) {
        float v = fabsf(aqo_bf16_to_f32(blk[e]));
        if (v > b) b = v;
      }
      float t = (b / 6.0f) * g_enc;
      uint8_t sf = aqo_e4m3_encode_satfinite(t);
      float sd = aqo_e4m3_decode(sf);
      scales[i * nblk + j] = sf;
      uint8_t q[16];
      if (sd == 0.0f) {
        memset(q, 0, sizeof q);
      } else {
        float r = g_enc / sd;
        for (int e = 0; e < 16; ++e)
          q[e] = aqo_e2m1_encode_satfinite(aqo_bf16_to_f32(blk[e]) * r);
      }
      uint8_t *dst = packed + i * (k / 2) + j * 8;
      for (int e = 0; e < 8; ++e)
        dst[e] = (uint8_t)(q[2 * e] | (q[2 * e + 1] << 4));
    }
  }
}

/* ------------------------------------------------------ device scale layout */

int64_t aqo_scale_layout_bytes(int64_t n, int64_t k) {
  int64_t tiles_n = (n + 15) / 16;
  int64_t tiles_k = (k + 127) / 128;
  return tiles_n * tiles_k * 128;
}

int64_t aqo_scale_layout_offset(int64_t row, int64_t block, int64_t k) {
  int64_t tiles_k = (k + 127) / 128;
  int64_t tn = row / 16, r = row % 16;
  int64_t tk = block / 8, j = block % 8;
  int64_t g = r % 8, h = r / 8;
  int64_t c = j / 2, p = j % 2;
  return (tn * tiles_k + tk) * 128 + (4 * g + c) * 4 + 2 * h + p;
}

void aqo_scales_to_device_layout(const uint8_t *canon, int64_t n, int64_t k,
                                 uint8_t *out) {
  memset(out, 0, (size_t)aqo_scale_layout_bytes(n, k));
  const int64_t nblk = k / 16;
  for (int64_t i = 0; i < n; ++i)
    for (int64_t j = 0; j < nblk; ++j)
      out[aqo_scale_layout_offset(i, j, k)] = canon[i * nblk + j];
}

/* ------------------------------------------------------------------ GEMV */

static double w_hat(const uint8_t *packed, const uint8_t *scales, double g_dec,
                    int64_t row, int64_t col, int64_t k) {
  uint8_t byte = packed[row * (k / 2) + col / 2];
  uint8_t nib = (col % 2) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
  double sd = (double)aqo_e4m3_decode(scales[row * (k / 16) + col / 16]);
  return (double)aqo_e2m1_decode(nib) * sd * g_dec;
}

/* [W] R10: fp64 accumulation, k ascending, of x times the dequantised
 * weight w_hat = e2m1(q) * sd * g_dec (each product exact in fp64). */
void aqo_gemv(const uint8_t *packed, const uint8_t *scales, float g_dec,
              const uint16_t *x, int64_t m, int64_t n, int64_t k,
              const int64_t *rows, int64_t nrows, double *y) {
  if (rows == NULL) nrows = n;
  for (int64_t t = 0; t < m; ++t) {
    for (int64_t i = 0; i < nrows; ++i) {
      int64_t row = rows ? rows[i] : i;
      double acc = 0.0;
      for (int64_t j = 0; j < k; ++j)
        acc += (double)aqo_bf16_to_f32(x[t * k + j]) *
               w_hat(packed, scales, (double)g_dec, row, j, k);
      y[t * nrows + i] = acc;
    }
  }
}

/* [U]: the plain dot product of each selected weight row with each token,
 * every bf16 value widened exactly and summed in fp64 in k order. */
void aqo_gemv_bf16(const uint16_t *w, const uint16_t *x, int64_t m, int64_t n, int64_t k,
                   const int64_t *rows, int64_t nrows, double *y) {
  if (rows == NULL) nrows = n;
  for (int64_t t = 0; t < m; ++t) {
    for (int64_t i = 0; i < nrows; ++i) {
      int64_t row = rows ? rows[i] : i;
      double acc = 0.0;
      for (int64_t j = 0; j < k; ++j)
        acc += (double)aqo_bf16_to_f32(x[t * k + j]) * (double)aqo_bf16_to_f32(w[row * k + j]);
      y[t * nrows + i] = acc;
    }
  }
}

/* [L]: the block product scaled per row, plus the rank-r term through the
 * r projections V^T x, each a plain fp64 sum. */
void aqo_gemv_lowrank(const uint8_t *packed, const uint8_t *scales, float g_dec, const float *s,
                      const uint16_t *U, const uint16_t *V, int64_t r, const uint16_t *x,
                      int64_t m, int64_t n, int64_t k, const int64_t *rows, int64_t nrows,
                      double *y) {
  if (rows == NULL) nrows = n;
  for (int64_t t = 0; t < m; ++t) {
    const uint16_t *xt = x + t * k;
    for (int64_t i = 0; i < nrows; ++i) {
      int64_t row = rows ? rows[i] : i;
      double base = 0.0;
      for (int64_t j = 0; j < k; ++j)
        base += (double)aqo_bf16_to_f32(xt[j]) * w_hat(packed, scales, (double)g_dec, row, j, k);
      double delta = 0.0;
      for (int64_t q = 0; q < r; ++q) {
        double vx = 0.0;
        for (int64_t j = 0; j < k; ++j)
          vx += (double)aqo_bf16_to_f32(V[j * r + q]) * (double)aqo_bf16_to_f32(xt[j]);
        delta += (double)aqo_bf16_to_f32(U[row * r + q]) * vx;
      }
      y[t * nrows + i] = (double)s[row] * base + delta;
    }
  }
}

/* [G] */
double aqo_gelu_tanh(double z) {
  const double c = sqrt(2.0 / 3.14159265358979323846);
  return 0.5 * z * (1.0 + tanh(c * (z + 0.044715 * z * z * z)));
}

/* [G]: the gate and up rows of output column j through the plain GEMV,
 * then gelu(gate) * up, all in fp64. */
void aqo_gemv_glu(const uint8_t *packed, const uint8_t *scales, float g_dec,
                  const uint16_t *x, int64_t m, int64_t n, int64_t k,
                  const int64_t *cols, int64_t ncols, double *h) {
  if (cols == NULL) ncols = n / 2;
  for (int64_t i = 0; i < ncols; ++i) {
    const int64_t j = cols ? cols[i] : i;
    const int64_t rows[2] = {(j / 8) * 16 + j % 8, (j / 8) * 16 + 8 + j % 8};
    double y[2];
    for (int64_t t = 0; t < m; ++t) {
      aqo_gemv(packed, scales, g_dec, x + t * k, 1, n, k, rows, 2, y);
      h[t * ncols + i] = aqo_gelu_tanh(y[0]) * y[1];
    }
  }
}

/* R9: every token row is quantised like a weight tensor of one row. */
int aqo_quantize_act(const uint16_t *x, int64_t m, int64_t k, uint8_t *packed,
                     uint8_t *scales, float *g_dec) {
  for (int64_t t = 0; t < m; ++t) {
    float ge, gd;
    int st = aqo_global_scales(aqo_amax_bf16(x + t * k, k), &ge, &gd);
    if (st != AQO_OK) return st;
    aqo_quantize_rows(x + t * k, 1, k, ge, packed + t * (k / 2),
                      scales + t * (k / 16));
    g_dec[t] = gd;
  }
  return AQO_OK;
}

void aqo_gemv_q(const uint8_t *w_packed, const uint8_t *w_scales, float w_gdec,
                const uint8_t *x_packed, const uint8_t *x_scales,
                const float *x_gdec, int64_t m, int64_t n, int64_t k,
                const int64_t *rows, int64_t nrows, double *y) {
  if (rows == NULL) nrows = n;
  for (int64_t t = 0; t < m; ++t) {
    for (int64_t i = 0; i < nrows; ++i) {
      int64_t row = rows ? rows[i] : i;
      double acc = 0.0;
      for (int64_t j = 0; j < k; ++j)
        acc += w_hat(x_packed, x_scales, (double)x_gdec[t], t, j, k) *
               w_hat(w_packed, w_scales, (double)w_gdec, row, j, k);
      y[t * nrows + i] = acc;
    }
  }
}

/* ------------------------------------------------------------ array forms */

void aqo_bf16_round_array(const float *in, int64_t count, uint16_t *out) {
  for (int64_t i = 0; i < count; ++i) out[i] = aqo_f32_to_bf16_rne(in[i]);
}
void aqo_e4m3_encode_array(const float *in, int64_t count, uint8_t *out) {
  for (int64_t i = 0; i < count; ++i) out[i] = aqo_e4m3_encode_satfinite(in[i]);
}
void aqo_e4m3_decode_array(const uint8_t *in, int64_t count, float *out) {
  for (int64_t i = 0; i < count; ++i) out[i] = aqo_e4m3_decode(in[i]);
}
void aqo_e2m1_encode_array(const float *in, int64_t count, uint8_t *out) {
  for (int64_t i = 0; i < count; ++i) out[i] = aqo_e2m1_encode_satfinite(in[i]);
}
void aqo_e2m1_decode_array(const uint8_t *in, int64_t count, float *out) {
  for (int64_t i = 0; i < count; ++i) out[i] = aqo_e2m1_decode(in[i]);
}
