/*
 * aq.h -- C ABI of the NVFP4 decode-projection library (libaq.so) for one
 * NVIDIA GB300 (sm_103a).
 *
 * What the library computes (sources are the AttnQuant / Weightless
 * documentation pages; page title, then section):
 *   - the effective weight of a theta bundle, W_eff = s*W0 + U*V^T, rebuilt
 *     once at load ("AttnQuant" landing page, "How it works"; Weightless
 *     "GPU and cache acceleration", "Precompute-outside (the fast path)");
 *   - its round-to-nearest NVFP4 quantisation: packed E2M1 nibbles, one
 *     E4M3 scale per 16 elements along K, one fp32 per-tensor scale
 *     (landing page "Results"; "GPU acceleration", "NVFP4 quantization";
 *     "Throughput", "What quantization actually saves");
 *   - the batch-1 / small-batch decode product y = x * W_hat^T streamed
 *     once per token, with Q/K/V and gate/up fused into single weights
 *     ("GPU acceleration", "Q/K/V fusion"; Weightless "Future work": a GEMV
 *     that dequantises in registers and streams at full HBM bandwidth);
 *   - the per-step stream of all projections of a decoder, one launch per
 *     fused projection ("GPU acceleration", "CUDA graph capture").
 *
 * Conventions shared by every entry point:
 *   - bf16 values are passed as uint16_t bit patterns.
 *   - Every pointer argument is DEVICE memory owned by the caller unless
 *     the comment says "host".  The library never allocates and never
 *     frees; it keeps no pointer after a call returns.
 *   - All work is asynchronous on the given stream (NULL = legacy default
 *     stream).  No call synchronises except aq_poll_device_status.
 *   - Arguments are validated on the host before any launch; a failed
 *     check launches nothing and returns an error code, with a message in
 *     aq_last_error().  Conditions only the device can see (a non-finite
 *     per-tensor amax, a bounded wait that gave up) are recorded in a
 *     device status word that aq_poll_device_status() reads and clears.
 *   - No C++ exception crosses this interface.
 *   - The stream type is the CUDA runtime's cudaStream_t (struct
 *     CUstream_st *); it is spelled here so the header needs no CUDA
 *     include.
 */
#ifndef AQ_H
#define AQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Only the entry points below are exported from libaq.so. */
#if defined(__GNUC__)
#define AQ_API __attribute__((visibility("default")))
#else
#define AQ_API
#endif

typedef struct CUstream_st *aq_stream_t;

typedef enum {
  AQ_OK = 0,
  AQ_ERR_INVALID_ARG = 1, /* null pointer, unknown enum value            */
  AQ_ERR_SHAPE = 2,       /* n, k, m or r outside the supported range     */
  AQ_ERR_ALIGNMENT = 3,   /* a pointer misses its stated alignment        */
  AQ_ERR_RANGE = 4,       /* per-tensor amax non-finite or too small      */
  AQ_ERR_UNSUPPORTED = 5, /* no sm_103 device, or path not available      */
  AQ_ERR_TIMEOUT = 6,     /* a bounded device-side wait gave up           */
  AQ_ERR_CUDA = 7,        /* a CUDA runtime call failed                   */
  AQ_ERR_WORKSPACE = 8    /* workspace missing, too small or misaligned   */
} aq_status;

/* An NVFP4 weight of shape [n, k] (n output rows, k input columns).  The
 * struct itself lives in host memory; its pointers are device memory.
 *   packed        n * k / 2 bytes, row-major; byte i of a row holds
 *                 element 2i in its low nibble and 2i+1 in its high
 *                 nibble; 16-byte aligned.
 *   scales        aq_scale_bytes(n, k) bytes of E4M3 block scales (one per
 *                 16 elements along k) in the device tile layout: tiles of
 *                 16 rows x 128 columns, tile (tn, tk) at byte
 *                 (tn * ceil(k/128) + tk) * 128; inside a tile, row
 *                 r = 8h + g and block j = 2c + p sit at byte
 *                 (4g + c) * 4 + 2h + p; padding bytes are zero.  One
 *                 32-bit word of a tile holds what one GEMV lane needs.
 *                 16-byte aligned.
 *   global_scale  one fp32: the per-tensor decode scale g_dec = amax/2688
 *                 (1 for an all-zero tensor).
 * A fused projection (Q/K/V, or gate and up) is one weight whose rows are
 * the row-wise concatenation of its parts, quantised with one per-tensor
 * scale. */
typedef struct {
  int32_t n;
  int32_t k;
  uint8_t *packed;
  uint8_t *scales;
  float *global_scale;
} aq_nvfp4_weight;

/* Shape limits: 1 <= n <= 2^24, 32 <= k <= 2^20, k % 32 == 0,
 * 0 <= r <= 64, 1 <= m <= AQ_MAX_M for the GEMV path. */
#define AQ_MAX_M 16
/* Tokens the block-scaled MMA path (AQ_PATH_MMA) serves per call. */
#define AQ_MAX_M_MMA 64

/* Bytes of the packed nibbles and of the scale layout of an [n, k] weight.
 * For n % 16 == 0 and k % 128 == 0 the two add up to 0.5625 * n * k.
 * Return 0 for shapes outside the limits. */
AQ_API size_t aq_packed_bytes(int32_t n, int32_t k);
AQ_API size_t aq_scale_bytes(int32_t n, int32_t k);

/* W_eff = bf16(s*W0 + U*V^T) ("How it works").  W0 [n, k], U [n, r],
 * V [k, r] bf16 row-major; s fp32 [n]; W_eff [n, k] bf16.  Per element the
 * rank-r term is summed first in fp32 (fused multiply-adds, r ascending,
 * starting from +0); if it is zero the value is the fp32 product s*W0,
 * otherwise one fused multiply-add s*W0 + delta; the fp32 result is rounded
 * to bf16 (nearest, ties to even).  So s = 1, U = V = 0 returns W0
 * bit-for-bit, -0 included.  r = 0 is allowed (U, V may then be NULL).
 * W0 and W_eff: 16-byte aligned; W_eff may not overlap the inputs. */
AQ_API aq_status aq_reconstruct(const uint16_t *W0, const float *s, const uint16_t *U,
                         const uint16_t *V, int32_t n, int32_t k, int32_t r,
                         uint16_t *W_eff, aq_stream_t stream);

/* Workspace of aq_quantize_nvfp4 and aq_reconstruct_quantize_nvfp4: at
 * least this many bytes, 256-byte aligned, device memory.  It must be
 * ZERO-FILLED once after allocation; every call leaves it zeroed (its
 * quantisation pass clears the amax and the grid-barrier words once all of
 * its CTAs have read them), so one workspace serves any sequence of calls on
 * one stream.  Calls that may run concurrently need separate workspaces.  A
 * call after which aq_poll_device_status reports AQ_ERR_TIMEOUT may leave
 * it dirty: zero it again before the next call. */
AQ_API size_t aq_quantize_workspace_bytes(void);

/* Round-to-nearest NVFP4 quantisation of a bf16 weight W [n, k] into *out
 * (whose n and k must equal the arguments).  Steps:
 *   amax = max |W|; g_enc = 2688/amax, g_dec = amax/2688 (1 and 1 if
 *   amax = 0); per 16-element block along k: b = max |w|,
 *   sf = E4M3((b/6)*g_enc) rounded to nearest even and saturated at 448,
 *   sd = decode(sf); if sd == 0 the block's nibbles are 0, else each
 *   nibble is E2M1(w * (g_enc/sd)), nearest even, saturated at 6, with the
 *   sign of the product kept even when the magnitude rounds to zero.
 * Writes out->packed, out->scales and *out->global_scale.  A non-finite
 * amax, or one so small that 2688/amax overflows, is caught on the device:
 * the outputs are then zero-filled, *global_scale is NaN, and the next
 * aq_poll_device_status() returns AQ_ERR_RANGE. */
AQ_API aq_status aq_quantize_nvfp4(const uint16_t *W, int32_t n, int32_t k,
                            const aq_nvfp4_weight *out, void *workspace,
                            size_t workspace_bytes, aq_stream_t stream);

/* The two steps above fused: W_eff is recomputed on the fly in both the
 * amax pass and the quantisation pass and never written to memory.  The
 * quantised bytes equal aq_reconstruct followed by aq_quantize_nvfp4. */
AQ_API aq_status aq_reconstruct_quantize_nvfp4(const uint16_t *W0, const float *s,
                                        const uint16_t *U, const uint16_t *V,
                                        int32_t n, int32_t k, int32_t r,
                                        const aq_nvfp4_weight *out,
                                        void *workspace, size_t workspace_bytes,
                                        aq_stream_t stream);

/* GEMV paths.  AQ_PATH_GEMV keeps the bf16 activations at full precision
 * and runs one of two kernels: the register-decode kernel (nibbles and
 * scales dequantised to f16 in registers, mma.sync), or for 1..5 tokens the
 * tcgen05 kernel, which hands the packed nibbles and E4M3 scales to the
 * block-scaled fp4 MMA unchanged and gives it each token's activations as
 * an exact-to-about-2^-19 sum of six NVFP4 terms.  AQ_PATH_AUTO and
 * AQ_PATH_GEMV pick the faster kernel for the shape (today the
 * register-decode one); the explicit choices exist for testing and
 * measurement. */
typedef enum {
  AQ_PATH_AUTO = 0,           /* GEMV for m <= AQ_MAX_M, MMA above           */
  AQ_PATH_GEMV = 1,           /* bf16 activations, kernel chosen by m        */
  AQ_PATH_MMA = 2,            /* activations quantised to NVFP4, tcgen05 MMA */
  AQ_PATH_GEMV_REGDECODE = 3, /* bf16 activations, register-decode kernel    */
  AQ_PATH_GEMV_TCGEN05 = 4    /* bf16 activations, tcgen05 kernel (m <= 5;
                                 AQ_ERR_UNSUPPORTED where it does not fit)  */
} aq_path;

/* Workspace of aq_gemv_nvfp4 / aq_decode_step_weights for a weight of
 * shape [n, k] and m tokens (1 <= m <= AQ_MAX_M_MMA): bytes, device memory,
 * 256-byte aligned, enough for every path that serves m tokens (for the
 * MMA path it also holds the quantised activations).  It must be
 * ZERO-FILLED once after allocation; every call leaves it in the state it
 * needs next, so one zeroed workspace serves any sequence of calls on one
 * stream.  Calls that may run concurrently need separate workspaces.  A
 * call after which aq_poll_device_status reports AQ_ERR_TIMEOUT may leave
 * it dirty: zero-fill it again before the next call. */
AQ_API size_t aq_gemv_workspace_bytes(int32_t n, int32_t k, int32_t m);

/* y[t, i] = bf16( sum_k x[t, k] * w_hat[i, k] ), w_hat = e2m1(q)*sd*g_dec,
 * fp32 accumulation ("Future work": a 4-bit GEMV at HBM bandwidth).  x [m, k]
 * bf16 and y [m, n] bf16 row-major, 16-byte aligned, y not overlapping x.
 * The result does not depend on timing (the split over the K axis is fixed
 * by (n, k) and its partial sums are added in a fixed order), and, within
 * one kernel, not on the rest of the batch: on the tcgen05 kernel each
 * token's output equals its m = 1 call bit for bit (m = 1..5); on the
 * register-decode kernel it is the same bits for every m = 2..16, while a
 * single token (m = 1) takes that kernel's one-token form, whose fp32 sums
 * run in a different order.  Every form meets the same tolerance against
 * the exact product. */
AQ_API aq_status aq_gemv_nvfp4(const aq_nvfp4_weight *w, const uint16_t *x, int32_t m,
                        uint16_t *y, aq_path path, void *workspace,
                        size_t workspace_bytes, aq_stream_t stream);

/* The block-scaled MMA path (AQ_PATH_MMA, and AQ_PATH_AUTO for m > AQ_MAX_M;
 * 1 <= m <= AQ_MAX_M_MMA).  AttnQuant docs, "Throughput", per-kernel
 * profile: the serving stack's NVFP4 projections are block-scaled fp4 GEMMs
 * that quantise the activations.  Each token row of x is first quantised on
 * its own exactly as aq_quantize_act_nvfp4 does (into the workspace); then
 *   y[t, i] = bf16( g_dec_w * g_dec_x[t] * sum_j sd_w[i, j] * sd_x[t, j]
 *                   * sum_{k in block j} e2m1(q_w[i, k]) * e2m1(q_x[t, k]) )
 * with fp32 accumulation on the tcgen05 tensor cores.  Outputs are within
 * the GEMV tolerance of the exact product of the two dequantised operands,
 * independent of timing, and each token's output does not depend on m.
 *
 * Per-row NVFP4 quantisation of activations (x [m, k] bf16 row-major,
 * 16-byte aligned): for each row its own amax, g_enc = 2688/amax,
 * g_dec[t] = amax/2688, and the block steps of aq_quantize_nvfp4.  packed
 * [m, k/2] (16-byte aligned), scales [m, k/16] E4M3 in canonical row-major
 * order (no tile layout), g_dec [m] fp32.  A row whose amax is non-finite or
 * too small is zero-filled, gets a NaN g_dec, and the next
 * aq_poll_device_status() returns AQ_ERR_RANGE.  1 <= m <= 2^20. */
AQ_API aq_status aq_quantize_act_nvfp4(const uint16_t *x, int32_t m, int32_t k,
                                       uint8_t *packed, uint8_t *scales, float *g_dec,
                                       aq_stream_t stream);

/* aq_gemv_nvfp4 without a workspace argument, for callers that cannot
 * allocate device memory: a plugin inside a host program that owns every
 * device allocation and forbids cudaMalloc once it is serving (cudaMalloc
 * may synchronise the device), or a binding that can pass buffers but not
 * create them.  The pages have no counterpart of this call; it exists for
 * such callers only.
 *
 * Arguments, results and errors are those of aq_gemv_nvfp4 on the
 * register-decode kernel, which computes every call: 1 <= m <= AQ_MAX_M,
 * and outputs equal aq_gemv_nvfp4 with AQ_PATH_GEMV_REGDECODE bit for bit.
 * AQ_PATH_MMA, AQ_PATH_GEMV_TCGEN05, and AQ_PATH_AUTO with m > AQ_MAX_M
 * (where aq_gemv_nvfp4 would take the MMA path) are rejected with
 * AQ_ERR_UNSUPPORTED.  The split-K
 * scratch is a fixed array of AQ_GEMV_NOALLOC_MAX_SCRATCH bytes inside the
 * library, in device memory, which every GPU that loads the library holds
 * until the process exits; nothing is allocated, on the device or the host.
 * A weight whose register-decode scratch on the current device exceeds that
 * size is rejected with AQ_ERR_WORKSPACE before any launch (that scratch
 * is 12 MiB plus 8 KiB x the number of 128-row blocks x the most CTAs that
 * share one of them, and never more than aq_gemv_workspace_bytes(n, k, m)).  The first call on each device
 * sets the array up synchronously (looks up its address and zero-fills
 * it), so that first call must come before any stream capture; the address
 * is kept for the life of the process, so the call must not be used across
 * a cudaDeviceReset.  Every call then clears, on `stream`, the
 * part of the array that has to start at zero, and launches the GEMV.
 * All calls on a device share the one array, which keeps the last call's
 * contents: calls whose kernels can overlap on the GPU (different streams,
 * different host threads) race on it and must be ordered by the caller. */
#define AQ_GEMV_NOALLOC_MAX_SCRATCH (32u << 20) /* bytes per device */
AQ_API aq_status aq_gemv_nvfp4_noalloc(const aq_nvfp4_weight *w, const uint16_t *x,
                                       int32_t m, uint16_t *y, aq_path path,
                                       aq_stream_t stream);

/* Flags of aq_decode_step_weights. */
#define AQ_STEP_PDL 1u /* programmatic dependent launch between projections */
#define AQ_STEP_REGDECODE 2u /* every projection on the register-decode kernel  */
#define AQ_STEP_TCGEN05 4u   /* the tcgen05 kernel wherever it serves the shape  */
#define AQ_STEP_MMA 8u       /* every projection on the block-scaled MMA path:
                                activations quantised to NVFP4 per row       */

/* One decode step's weight stream: for p = 0 .. n_proj-1 in order,
 * y[p] = GEMV(w[p], x[p]) with m tokens, all on one stream, one launch per
 * projection.  w, x and y are HOST arrays of n_proj entries; the weights
 * and activation buffers they point to are device memory.  Projection p+1
 * reads its x only after projection p has completed (stream order, or with
 * AQ_STEP_PDL a programmatic wait inside the kernel after it has started
 * fetching its weights).  workspace must hold aq_gemv_workspace_bytes for
 * the largest projection and be zero-filled once.  Safe to record into a
 * CUDA graph. */
AQ_API aq_status aq_decode_step_weights(const aq_nvfp4_weight *w, int32_t n_proj,
                                 const uint16_t *const *x, uint16_t *const *y,
                                 int32_t m, uint32_t flags, void *workspace,
                                 size_t workspace_bytes, aq_stream_t stream);

/* GEMV of a weight kept in bf16: the projections the method leaves
 * unquantised -- the tied lm_head / embedding, and the attention projections
 * when they are excluded from quantisation (AttnQuant docs, "GPU
 * acceleration", "Where GPU time goes": these bf16 families stream beside
 * the NVFP4 MLP in every decode step; "NVFP4 quantization": 2.82 GB of bf16
 * embedding / lm_head on the 31B model).
 *
 * y[t, i] = bf16( sum_k x[t, k] * w[i, k] ), fp32 accumulation.  w [n, k]
 * bf16 row-major (device, caller-owned, read only), 1 <= n <= 2^24,
 * 8 <= k <= 2^20 with k % 8 == 0; x [m, k] and y [m, n] bf16 row-major,
 * 1 <= m <= AQ_MAX_M; w, x, y 16-byte aligned, y not overlapping x or w.
 * The split over K is fixed by (n, k) and the device, so the result does
 * not depend on timing, and each token's output equals the m = 1 call bit
 * for bit.  flags: 0 or AQ_STEP_PDL (the kernel waits for the previous
 * launch on the stream programmatically, after it has started fetching
 * weights).  workspace: aq_gemv_bf16_workspace_bytes(n, k, m) bytes of
 * device memory, 256-byte aligned, zero-filled once, with the same
 * contract as the NVFP4 GEMV's (and interchangeable with it: one workspace
 * of the larger size serves both).  Errors: AQ_ERR_SHAPE, AQ_ERR_ALIGNMENT,
 * AQ_ERR_INVALID_ARG, AQ_ERR_WORKSPACE before any launch; AQ_ERR_TIMEOUT
 * through aq_poll_device_status. */
AQ_API size_t aq_gemv_bf16_workspace_bytes(int32_t n, int32_t k, int32_t m);

/* The runtime low-rank GEMV: the projection evaluated from its theta bundle
 * without rebuilding the weight (AttnQuant docs, "Throughput", "The runtime
 * reconstruction path does not reach dense parity", and "GPU acceleration",
 * "How the pieces fit": one kernel fuses the shared-block dot product with
 * the low-rank delta; landing page, "How it works": W_eff = s*W0 + U V^T),
 * with the shared block W0 quantised to NVFP4:
 *
 *   y[t, i] = bf16( s[i] * (g_dec * acc[t, i]) + sum_q U[i, q] * v[t, q] ),
 *   acc[t, i] = sum_k x[t, k] * e2m1(q0[i, k]) * sd0[i, k/16] (fp32, as in
 *   aq_gemv_nvfp4 on the register-decode kernel), v = V^T x in fp32.
 *
 * w0 as for aq_gemv_nvfp4 (it may be shared by every projection of a band);
 * s fp32 [n]; U bf16 [n, r] and V bf16 [k, r] row-major (device, NULL when
 * r == 0), 0 <= r <= AQ_LOWRANK_MAX_R; x, y, m as for aq_gemv_nvfp4 with
 * 1 <= m <= AQ_MAX_M.  Two launches on `stream`: v = V^T x into the
 * workspace, then the GEMV, chained with programmatic dependent launch;
 * flags 0 or AQ_STEP_PDL (the first launch waits for the previous work on
 * the stream programmatically).  With s = 1 and r = 0 the result equals
 * aq_gemv_nvfp4 with AQ_PATH_GEMV_REGDECODE bit for bit.  workspace:
 * aq_gemv_lowrank_workspace_bytes(n, k, m, r) bytes, 256-byte aligned,
 * zero-filled once; its first aq_gemv_workspace_bytes(n, k, m) bytes follow
 * the GEMV workspace contract, v lives after them.  Errors as for
 * aq_gemv_nvfp4. */
#define AQ_LOWRANK_MAX_R 16

/* Per-segment tensor scales for a fused weight (the quality-preserving
 * form of the fusion: each sub-projection -- q, k, v or gate, up -- keeps
 * the per-tensor scale it would have on its own; AttnQuant docs, "GPU
 * acceleration", "NVFP4 quantization": checkpoints quantised projection by
 * projection; "Q/K/V fusion" for the fused weight itself).
 *
 * Segments: 1 <= nseg <= AQ_MAX_SEGMENTS, seg_end a HOST array of strictly
 * increasing row ends, seg_end[nseg-1] == n, every segment start a multiple
 * of 16 (so each segment owns whole scale tiles).  Segment s is rows
 * [seg_end[s-1], seg_end[s]) (seg_end[-1] = 0).
 *
 * aq_quantize_nvfp4_segments: each segment of W [n, k] quantised exactly as
 * aq_quantize_nvfp4 would quantise it alone (its own amax, g_enc, g_dec),
 * written at its rows of out->packed / out->scales; out->global_scale
 * points to nseg floats, g_dec of segment s at index s.
 * aq_gemv_nvfp4_segments: y[t, i] = bf16(g_dec[segment(i)] * acc[t, i]) on
 * the register-decode kernel (acc as in aq_gemv_nvfp4); x, y, m (<=
 * AQ_MAX_M), flags (0 or AQ_STEP_PDL), workspace and errors as there.  With
 * one segment both equal their plain counterparts bit for bit. */
#define AQ_MAX_SEGMENTS 8
AQ_API aq_status aq_quantize_nvfp4_segments(const uint16_t *W, int32_t n, int32_t k,
                                            int32_t nseg, const int32_t *seg_end,
                                            const aq_nvfp4_weight *out, void *workspace,
                                            size_t workspace_bytes, aq_stream_t stream);
AQ_API aq_status aq_gemv_nvfp4_segments(const aq_nvfp4_weight *w, int32_t nseg,
                                        const int32_t *seg_end, const uint16_t *x, int32_t m,
                                        uint16_t *y, uint32_t flags, void *workspace,
                                        size_t workspace_bytes, aq_stream_t stream);

/* Fused gate+up with its activation in the epilogue (the gated MLP's first
 * half in one pass: the pages count 0.44 ms of elementwise work per 31B
 * step beside the GEMVs, AttnQuant docs, "Throughput", where the step's
 * time goes; and the gate+up fusion itself, "GPU acceleration", "Q/K/V
 * fusion" and Weightless docs, "Future work", "Gate/up fusion").
 *
 *   h[t, j] = bf16( gelu(g_dec * acc[t, gate j]) * (g_dec * acc[t, up j]) ),
 *   gelu(z) = 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))) in fp32,
 *
 * acc as in aq_gemv_nvfp4 on the register-decode kernel.  The weight's rows
 * interleave gate and up in groups of 8 -- rows 16 j' .. 16 j'+7 are gate
 * rows 8 j' .. 8 j'+7, rows 16 j'+8 .. 16 j'+15 the matching up rows -- so
 * n = 2 f is a multiple of 16 and h is [m, f] bf16 (16-byte aligned).
 * aq_interleave_gate_up produces that order from the row-concatenated
 * [gate; up] bf16 weight before quantisation (a row permutation: the
 * tensor's amax, so its per-tensor scale, and every row's bytes are those
 * of the concatenated weight).  m, x, flags (0 or AQ_STEP_PDL), workspace
 * (aq_gemv_workspace_bytes) and errors as for aq_gemv_nvfp4. */
AQ_API aq_status aq_interleave_gate_up(const uint16_t *w, int32_t f, int32_t k, uint16_t *out,
                                       aq_stream_t stream);
AQ_API aq_status aq_gemv_glu_nvfp4(const aq_nvfp4_weight *w, const uint16_t *x, int32_t m,
                                   uint16_t *h, uint32_t flags, void *workspace,
                                   size_t workspace_bytes, aq_stream_t stream);
AQ_API size_t aq_gemv_lowrank_workspace_bytes(int32_t n, int32_t k, int32_t m, int32_t r);
AQ_API aq_status aq_gemv_lowrank_nvfp4(const aq_nvfp4_weight *w0, const float *s,
                                       const uint16_t *U, const uint16_t *V, int32_t r,
                                       const uint16_t *x, int32_t m, uint16_t *y,
                                       uint32_t flags, void *workspace,
                                       size_t workspace_bytes, aq_stream_t stream);
AQ_API aq_status aq_gemv_bf16(const uint16_t *w, int32_t n, int32_t k, const uint16_t *x,
                              int32_t m, uint16_t *y, uint32_t flags, void *workspace,
                              size_t workspace_bytes, aq_stream_t stream);

/* The decode step's weight stream as ONE persistent kernel ("GPU
 * acceleration", "CUDA graph capture": replay the step without per-kernel
 * dispatch; "Q/K/V fusion": one weight read per fused projection).
 *
 * aq_step_plan_create validates the projections exactly like
 * aq_decode_step_weights, encodes their tensor maps and stream-K
 * partitions, and uploads them (synchronously, cudaMemcpy) into `plan`:
 * device memory of aq_step_plan_bytes(n_proj) bytes, 128-byte aligned,
 * owned by the caller and read by every aq_step_run until the caller frees
 * it.  The weight, x and y pointers are baked into the plan, so the buffers
 * must stay allocated and keep their addresses.  *workspace_bytes receives
 * the workspace size aq_step_run needs; that workspace must be zero-filled
 * once after allocation and is left ready for the next run.
 *
 * aq_step_run computes, for p = 0 .. n_proj-1 in order,
 * y[p] = GEMV(w[p], x[p]) with the m tokens the plan was made for, in one
 * cooperative launch on `stream`: every CTA streams the weights of all
 * projections back to back, and before reading x[p] it waits (grid-wide,
 * bounded) until every output of projection p-1 is written.  Results equal
 * the per-projection calls to within the GEMV tolerance (the split over K
 * can differ).  A plan, m or workspace that does not match is reported by
 * the next aq_poll_device_status() as AQ_ERR_INVALID_ARG.  Safe to record
 * into a CUDA graph; runs that may overlap need separate workspaces. */
AQ_API size_t aq_step_plan_bytes(int32_t n_proj);
AQ_API aq_status aq_step_plan_create(const aq_nvfp4_weight *w, int32_t n_proj,
                                     const uint16_t *const *x, uint16_t *const *y, int32_t m,
                                     void *plan, size_t plan_bytes, size_t *workspace_bytes);
AQ_API aq_status aq_step_run(const void *plan, int32_t m, void *workspace,
                             size_t workspace_bytes, aq_stream_t stream);

/* Test helper: the scales of w rewritten in canonical row-major order
 * [n, k/16] into canon (device, n*k/16 bytes). */
AQ_API aq_status aq_scales_to_canonical(const aq_nvfp4_weight *w, uint8_t *canon,
                                 aq_stream_t stream);

/* Test hook of the failure path: one kernel runs the GEMV kernels' bounded
 * ring wait (the same device function) against a barrier that nothing
 * completes, with at most `polls` polls (1 <= polls <= 2^20).  It gives up,
 * records AQ_ERR_TIMEOUT in the device status word and returns; the next
 * aq_poll_device_status reports AQ_ERR_TIMEOUT and the context stays
 * usable.  No memory is touched.  The pages have no counterpart; it exists
 * so the timeout path can be exercised without a fault. */
AQ_API aq_status aq_selftest_timeout(uint32_t polls, aq_stream_t stream);

/* Synchronise `stream`, read the device status word of the current device
 * and clear it.  Returns AQ_OK, AQ_ERR_RANGE or AQ_ERR_TIMEOUT (the first
 * condition recorded since the last poll), or AQ_ERR_CUDA. */
AQ_API aq_status aq_poll_device_status(aq_stream_t stream);

/* Message of the last error returned on the calling host thread ("" if
 * none).  The string stays valid until the thread's next failing call. */
AQ_API const char *aq_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
AQ_API int32_t aq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* AQ_H */
