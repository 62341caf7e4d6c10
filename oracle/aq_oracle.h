/*
 * aq_oracle.h -- CPU oracle for the NVFP4 decode-projection path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load this library.  The
 * CUDA library never includes, links or calls anything here, and nothing
 * here includes a CUDA header: the two implementations share no code.
 *
 * Plain C11, single thread, no vectorisation tricks.  Every float32 step is
 * one IEEE-754 binary32 operation rounded to nearest-even (the build uses
 * -ffp-contract=off and no fast-math), so a reader can check each function
 * against the definition it cites.
 *
 * Sources (page title, section):
 *   [H]  AttnQuant docs, landing page, "How it works": each projection is a
 *        theta bundle (shared block W0, per-row scale s, low-rank U, V); the
 *        effective weight W_eff = s*W0 + U*V^T is rebuilt once at load.
 *   [R]  AttnQuant docs, landing page, "Results" ("Full coverage, no
 *        calibration"): quantisation is round-to-nearest, no calibration.
 *   [Q]  AttnQuant docs, "GPU acceleration", "NVFP4 quantization": the
 *        quantised weight is packed uint8 nibbles plus float8 block scales.
 *   [B]  AttnQuant docs, "Throughput", "What quantization actually saves":
 *        0.5625 B/element = 0.5 B packed weight + one float8_e4m3fn scale
 *        per 16 elements.
 *   [P]  AttnQuant docs, "Throughput", "Where the throughput comes from" and
 *        landing page "Where the speed comes from": at the passthrough
 *        setting the decomposition rebuilds the original weight bit-for-bit.
 *   [W]  Weightless docs, "GPU and cache acceleration", "Future work": a
 *        GEMV that dequantises 4-bit weights in registers.
 *   [L]  AttnQuant docs, "Throughput", "The runtime reconstruction path does
 *        not reach dense parity", and "GPU acceleration", "How the pieces
 *        fit" (the custom op that fuses the shared-block dot product and the
 *        low-rank delta): the runtime path evaluates s*(W0 x) + U (V^T x)
 *        instead of a rebuilt weight.
 *   [G]  AttnQuant docs, "Throughput" (the step's elementwise work beside
 *        the GEMVs) and Weightless docs, "Future work" ("Gate/up fusion"):
 *        the gated MLP's h = act(gate) * up; act read as the tanh form of
 *        GELU (the design notes' reading R15).
 *   [U]  AttnQuant docs, "GPU acceleration", "Where GPU time goes": the
 *        attention projections (when left unquantised) and the tied
 *        lm_head / embedding are bf16 weights streamed by plain GEMVs.
 *   [F]  NVFP4 format: E2M1 element grid {0, +-0.5, +-1, +-1.5, +-2, +-3,
 *        +-4, +-6}; E4M3 (float8_e4m3fn: bias 7, max 448, no infinities)
 *        block scale per 16 elements; one fp32 per-tensor scale.  The
 *        element and scale encodings are those of the OCP Microscaling
 *        Formats specification (FP4 E2M1, FP8 E4M3).
 *
 * Readings where the pages are silent (each is listed with its reason in
 * the design notes): R1 reconstruction order, R2 per-tensor constant 2688,
 * R3 block-scale operation order, R4 satfinite / zero scale, R5 element
 * rounding ties-to-even with signed zero, R6 nibble order, R7 device scale
 * layout, R9 per-row activation quantisation, R10 GEMV acceptance rule.
 */
#ifndef AQ_ORACLE_H
#define AQ_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define AQO_OK 0
#define AQO_ERR_RANGE 4 /* non-finite amax, or amax so small 2688/amax overflows */

/* bf16 <-> fp32.  bf16 values travel as their uint16 bit patterns. */
float aqo_bf16_to_f32(uint16_t h);
uint16_t aqo_f32_to_bf16_rne(float f);

/* [F] E4M3 (float8_e4m3fn) scale: decode, and encode with round-to-nearest-
 * even and saturation to +-448 (R4).  NaN encodes to 0x7F. */
float aqo_e4m3_decode(uint8_t code);
uint8_t aqo_e4m3_encode_satfinite(float t);

/* [F] E2M1 element nibble: decode, and encode with round-to-nearest-even,
 * saturation to +-6 and the sign kept on values that round to zero (R5). */
float aqo_e2m1_decode(uint8_t nibble);
uint8_t aqo_e2m1_encode_satfinite(float v);

/* [H] R1: W_eff[n,k] = bf16( s[n]*W0[n,k] + sum_r U[n,r]*V[k,r] ).
 * W0 [n,k], U [n,r], V [k,r] bf16 row-major; s fp32 [n]; W_eff [n,k]. */
void aqo_reconstruct(const uint16_t *W0, const float *s, const uint16_t *U,
                     const uint16_t *V, int64_t n, int64_t k, int64_t r,
                     uint16_t *W_eff);

/* max |w| over count bf16 values, as fp32 (exact).  NaN if any is NaN. */
float aqo_amax_bf16(const uint16_t *W, int64_t count);

/* R2: g_enc = 2688/amax, g_dec = amax/2688 (two IEEE divisions);
 * amax == 0 gives g_enc = g_dec = 1.  Returns AQO_ERR_RANGE for a
 * non-finite or negative amax, or one so small that g_enc overflows. */
int aqo_global_scales(float amax, float *g_enc, float *g_dec);

/* [Q][R][F] R3-R6: quantise `rows` rows of W [rows, k] (k % 16 == 0) with
 * the per-tensor encode scale g_enc.  packed [rows, k/2] (element 2i in the
 * low nibble of byte i), scales [rows, k/16] E4M3 in canonical row-major
 * order. */
void aqo_quantize_rows(const uint16_t *W, int64_t rows, int64_t k, float g_enc,
                       uint8_t *packed, uint8_t *scales);

/* R7 device scale layout: tiles of 16 rows x 128 columns (8 blocks), tile
 * (tn, tk) at byte ((tn * ceil(k/128)) + tk) * 128; inside a tile, row
 * r = 8h + g and block j = 2c + p live at byte (4g + c)*4 + 2h + p.  Bytes
 * of rows >= n or blocks >= k/16 are zero padding. */
int64_t aqo_scale_layout_bytes(int64_t n, int64_t k);
int64_t aqo_scale_layout_offset(int64_t row, int64_t block, int64_t k);
void aqo_scales_to_device_layout(const uint8_t *canon, int64_t n, int64_t k,
                                 uint8_t *out);

/* [W] R10: y[m, i] = sum_k x[m,k] * w_hat[rows[i], k] in fp64, k ascending,
 * with w_hat = e2m1(q) * decode(scale) * g_dec.  x bf16 [m, k]; packed and
 * canonical scales cover all n rows; `rows` (nrows entries) selects the
 * rows to evaluate, or NULL for all n rows in order (then nrows = n).
 * y is [m, nrows] row-major. */
void aqo_gemv(const uint8_t *packed, const uint8_t *scales, float g_dec,
              const uint16_t *x, int64_t m, int64_t n, int64_t k,
              const int64_t *rows, int64_t nrows, double *y);

/* R9: quantise each token row of x [m, k] on its own (own amax, own g_enc,
 * own block scales): packed [m, k/2], scales [m, k/16] canonical, g_dec [m].
 * Returns AQO_ERR_RANGE if any row's amax is out of range. */
int aqo_quantize_act(const uint16_t *x, int64_t m, int64_t k, uint8_t *packed,
                     uint8_t *scales, float *g_dec);

/* Block-scaled product of a quantised weight and quantised activations:
 * y[m, i] = sum_k x_hat[m,k] * w_hat[rows[i],k] in fp64, k ascending. */
void aqo_gemv_q(const uint8_t *w_packed, const uint8_t *w_scales, float w_gdec,
                const uint8_t *x_packed, const uint8_t *x_scales,
                const float *x_gdec, int64_t m, int64_t n, int64_t k,
                const int64_t *rows, int64_t nrows, double *y);

/* [U] GEMV of a bf16 weight: y[m, i] = sum_k x[m,k] * w[rows[i],k] in
 * fp64, k ascending, both operands bf16 [.., k] row-major.  rows / nrows
 * as in aqo_gemv. */
void aqo_gemv_bf16(const uint16_t *w, const uint16_t *x, int64_t m, int64_t n, int64_t k,
                   const int64_t *rows, int64_t nrows, double *y);

/* [L] [H] runtime low-rank GEMV with a quantised shared block:
 * y[m, i] = s[i] * sum_k x[m,k] * w0_hat[i,k]
 *         + sum_r U[i,r] * (sum_k V[k,r] * x[m,k]),
 * every sum in fp64 in index order, w0_hat = e2m1(q) * sd * g_dec of the
 * quantised W0 (packed, canonical scales); s fp32 [n], U bf16 [n, r],
 * V bf16 [k, r], x bf16 [m, k]; r may be 0.  rows / nrows as in aqo_gemv. */
void aqo_gemv_lowrank(const uint8_t *packed, const uint8_t *scales, float g_dec, const float *s,
                      const uint16_t *U, const uint16_t *V, int64_t r, const uint16_t *x,
                      int64_t m, int64_t n, int64_t k, const int64_t *rows, int64_t nrows,
                      double *y);

/* [G] the tanh form of GELU in fp64:
 * 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))). */
double aqo_gelu_tanh(double z);

/* [G] fused gate+up with the activation applied: the weight's rows
 * interleave gate and up in groups of 8 (row 16j'+i gate, 16j'+8+i up, of
 * output column j = 8j'+i); h[m, c] = gelu(y_gate) * y_up with y the fp64
 * GEMV (aqo_gemv) of those two rows, for the selected output columns
 * `cols` (ncols entries, or NULL for all n/2 in order).  h [m, ncols]. */
void aqo_gemv_glu(const uint8_t *packed, const uint8_t *scales, float g_dec,
                  const uint16_t *x, int64_t m, int64_t n, int64_t k,
                  const int64_t *cols, int64_t ncols, double *h);

/* Element-wise array forms of the five scalar conversions above (one call
 * per element, in order), so tests can sweep many values cheaply. */
void aqo_bf16_round_array(const float *in, int64_t count, uint16_t *out);
void aqo_e4m3_encode_array(const float *in, int64_t count, uint8_t *out);
void aqo_e4m3_decode_array(const uint8_t *in, int64_t count, float *out);
void aqo_e2m1_encode_array(const float *in, int64_t count, uint8_t *out);
void aqo_e2m1_decode_array(const uint8_t *in, int64_t count, float *out);

#ifdef __cplusplus
}
#endif
#endif /* AQ_ORACLE_H */
