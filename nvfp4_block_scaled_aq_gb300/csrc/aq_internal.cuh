// aq_internal.cuh -- device helpers and internal host declarations shared by
// the kernels of libaq.so.  Written for sm_103a only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cuda.h>

#include "../../include/aq.h"

namespace aq {

// ------------------------------------------------------------ status word
// One 32-bit word per device records the first device-detected condition
// since the last poll (0 = none).  Kernels receive its address.
enum : unsigned { kDevOk = 0, kDevRange = 1, kDevTimeout = 2, kDevBadPlan = 3 };

__device__ __forceinline__ void raise_status(unsigned *status, unsigned code) {
  atomicCAS(status, 0u, code);
}

// ------------------------------------------------------------ constants
constexpr int kTileRows = 16;    // rows of a scale tile / GEMV warp tile
constexpr int kTileCols = 128;   // columns of a scale tile (8 blocks)
constexpr int kBlock = 16;       // elements per E4M3 block scale
constexpr float kGlobalMax = 2688.0f;  // 6 (largest E2M1) * 448 (largest E4M3)

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) {
  return (a + b - 1) / b;
}

// Byte offset of block `blk` of row `row` in the scale tile layout.
__host__ __device__ __forceinline__ int64_t scale_offset(int64_t row, int64_t blk,
                                                         int64_t k) {
  const int64_t tiles_k = ceil_div(k, kTileCols);
  const int64_t tn = row >> 4, r = row & 15;
  const int64_t tk = blk >> 3, j = blk & 7;
  return (tn * tiles_k + tk) * 128 + ((r & 7) * 4 + (j >> 1)) * 4 + (r >> 3) * 2 +
         (j & 1);
}

// ------------------------------------------------------------ bf16 bits
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

// ------------------------------------------------------------ FP8 / FP4 cvt
// Two fp32 -> e4m3x2 (nearest even, saturate to +-448): `hi` lands in the
// upper byte.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// e4m3x2 (16 bits) -> f16x2 (exact): the low byte goes to the low half.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// Two fp32 -> one byte of two E2M1 codes (nearest even, saturate to +-6,
// sign kept): `hi` goes to the high nibble.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float hi, float lo) {
  uint32_t r;
  asm("{ .reg .b8 t;\n"
      "  cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n"
      "  cvt.u32.u8 %0, t; }"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Four E2M1 pairs of a 32-bit word -> four f16x2 (exact): byte i of `w`
// (elements 2i, 2i+1) becomes out[i] with element 2i in the low half.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t out[4]) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n"
      "  mov.b32 {b0, b1, b2, b3}, %4;\n"
      "  cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      "  cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "  cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      "  cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(w));
}

// Low f16 half of a pair -> fp32 (exact).
__device__ __forceinline__ float f16_lo_to_f32(uint32_t h2) {
  float f;
  asm("{ .reg .b16 l, h;\n"
      "  mov.b32 {l, h}, %1;\n"
      "  cvt.f32.f16 %0, l; }"
      : "=f"(f)
      : "r"(h2));
  return f;
}

// High f16 half of a pair -> fp32 (exact).
__device__ __forceinline__ float f16_hi_to_f32(uint32_t h2) {
  float f;
  asm("{ .reg .b16 l, h;\n"
      "  mov.b32 {l, h}, %1;\n"
      "  cvt.f32.f16 %0, h; }"
      : "=f"(f)
      : "r"(h2));
  return f;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Two fp32 -> f16x2 (nearest even); `hi` lands in the upper half.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float hi, float lo) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ------------------------------------------------------------ tensor core
// D = A(16x16 f16, row) * B(16x8 f16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float d[4], const uint32_t a[4],
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------ memory
// Streaming 16-byte load that bypasses L1 (weights are read once).
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_stream_u32(const void *p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// ------------------------------------------------------------ PDL
// Programmatic dependent launch: let the next kernel in the stream start
// launching, and wait until the previous kernel's memory is visible.
// Both are no-ops when the launch carries no programmatic dependency.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace aq

// ------------------------------------------------------------ host side
namespace aq {

struct DeviceInfo {
  int ordinal;
  int sms;
  int cc_major, cc_minor;
  size_t smem_optin;
  unsigned *status;  // device address of the status word
};

// Per-device facts, resolved once per device (thread-safe).  Returns
// nullptr and sets the last error when the current device is unusable.
const DeviceInfo *device_info();

aq_status set_error(aq_status st, const char *fmt, ...);
aq_status cuda_error(cudaError_t e, const char *what);

// Launchers implemented by the kernel translation units.  Arguments are
// validated by the caller.
cudaError_t launch_reconstruct(const uint16_t *W0, const float *s, const uint16_t *U,
                               const uint16_t *V, int n, int k, int r, uint16_t *W_eff,
                               cudaStream_t st);
cudaError_t launch_quantize(const uint16_t *W, const float *s, const uint16_t *U,
                            const uint16_t *V, int r, bool fused, int n, int k,
                            const aq_nvfp4_weight &out, void *ws, const DeviceInfo &dev,
                            cudaStream_t st);
// Per-row NVFP4 quantisation of activations (quantize.cu); scales row-major
// with a pitch of scale_pitch bytes.  pdl: launched as a programmatic
// dependent of the previous kernel on the stream (it waits for it before
// reading x); either way the kernel lets its own dependents start early.
cudaError_t launch_act_quant(const uint16_t *x, int m, int k, uint8_t *packed, uint8_t *scales,
                             int scale_pitch, float *g_dec, const DeviceInfo &dev,
                             cudaStream_t st, bool pdl = false);
cudaError_t launch_scales_to_canonical(const aq_nvfp4_weight &w, uint8_t *canon,
                                       cudaStream_t st);
cudaError_t launch_interleave_gate_up(const uint16_t *w, int f, int k, uint16_t *out,
                                      cudaStream_t st);

struct GemvPlan {
  int64_t row_blocks;  // ceil(n / rows_per_block)
  int64_t k_tiles;     // ceil(k / 128)
  int64_t units;       // work units per row block
  int64_t total;       // row_blocks * units
  int grid;            // persistent CTAs
  int max_contrib;     // most CTAs sharing one row block
};
// Split-K tickets per row block at the start of a GEMV workspace (one per
// 16-row group of the register-decode kernel).
constexpr int kTicketsPerRowBlock = 8;
// Row groups of 16 rows per CTA of the register-decode GEMV (the single
// calls and the decode step): 8 (two CTAs per SM, 128-row units) or 16 (one
// CTA per SM, 256-row units).  Measured on the ~31B step at m = 1: 3.26 ms
// with 8, 3.30 ms with 16 (per-projection launches); the persistent step
// 3.80 / 3.77 ms.
constexpr int kGemvRG = 8;
GemvPlan plan_gemv(int n, int k, const DeviceInfo &dev, int rg);
size_t gemv_workspace_bytes(int n, int k, const DeviceInfo &dev);
size_t gemv_regdecode_workspace_bytes(int n, int k, const DeviceInfo &dev);
// `next`, when given, is the projection launched after this one on the same
// stream: the kernel prefetches the first weight units of it into L2.
cudaError_t launch_gemv(const aq_nvfp4_weight &w, const uint16_t *x, int m, uint16_t *y,
                        void *ws, bool pdl, const DeviceInfo &dev, cudaStream_t st,
                        const aq_nvfp4_weight *next = nullptr);
// The tcgen05 kernel (tc_gemv.cu): its plan, whether it serves a shape for
// m tokens, its workspace, and its launch.
GemvPlan plan_gemv_tc(int n, int k, const DeviceInfo &dev);
bool tc_eligible(int n, int k, int m, const DeviceInfo &dev);
size_t gemv_tc_workspace_bytes(int n, int k, const DeviceInfo &dev);
cudaError_t launch_gemv_tc(const aq_nvfp4_weight &w, const uint16_t *x, int m, uint16_t *y,
                           void *ws, bool pdl, const DeviceInfo &dev, cudaStream_t st);
// The block-scaled MMA path (mma_gemm.cu): workspace layout for m tokens,
// eligibility, and the launch of activation quantisation + MMA kernel.
struct MmaWorkspace {
  int slots;                 // partial-sum token slots per row
  int scale_pitch;           // bytes per row of the activation scales
  size_t partial_off, xq_off, xs_off, xg_off, bytes;
};
MmaWorkspace mma_workspace(int n, int k, int m, const DeviceInfo &dev);
bool mma_eligible(int n, int k, int m, const DeviceInfo &dev);
cudaError_t launch_mma(const aq_nvfp4_weight &w, const uint16_t *x, int m, uint16_t *y, void *ws,
                       bool pdl, const DeviceInfo &dev, cudaStream_t st);
// Tensor maps of quantised activations: nibbles [m, k/2] in boxes of
// 128 B x n_box rows (128-byte swizzle) and scales [m rows, pitch bytes] in
// boxes of 16 B x n_box rows (gemv.cu).
bool encode_act_maps(const uint8_t *xq, const uint8_t *xs, int m, int k, int scale_pitch,
                     int n_box, CUtensorMap *tm_x, CUtensorMap *tm_xs);
// The bf16 GEMV (gemv_bf16.cu): plan, workspace and launch.
GemvPlan plan_gemv_bf16(int n, int k, const DeviceInfo &dev);
size_t gemv_bf16_workspace_bytes(int n, int k, const DeviceInfo &dev);
cudaError_t launch_gemv_bf16(const uint16_t *w, int n, int k, const uint16_t *x, int m,
                             uint16_t *y, void *ws, bool pdl, const DeviceInfo &dev,
                             cudaStream_t st);
// Self-test of the bounded-wait error path (gemv.cu).
cudaError_t launch_selftest_wait(unsigned polls, const DeviceInfo &dev, cudaStream_t st);
// Register-decode kernel only (gemv.cu).
// The runtime low-rank epilogue terms (see Proj in gemv_core.cuh).
struct LowRank {
  const float *s;
  const uint16_t *u;
  const float *t;
  int r;
};
cudaError_t launch_gemv_regdecode(const aq_nvfp4_weight &w, const uint16_t *x, int m,
                                  uint16_t *y, void *ws, bool pdl, const DeviceInfo &dev,
                                  cudaStream_t st, const aq_nvfp4_weight *next = nullptr,
                                  const LowRank *lr = nullptr, bool glu = false,
                                  int nseg = 0, const int32_t *seg_end = nullptr);
// y = s * (W0_hat x) + U (V^T x) (lowrank.cu): workspace and launch.
size_t gemv_lowrank_workspace_bytes(int n, int k, int m, int r, const DeviceInfo &dev);
cudaError_t launch_gemv_lowrank(const aq_nvfp4_weight &w0, const float *s, const uint16_t *U,
                                const uint16_t *V, int r, const uint16_t *x, int m,
                                uint16_t *y, void *ws, bool pdl, const DeviceInfo &dev,
                                cudaStream_t st);
cudaError_t launch_gemv_uncached(const aq_nvfp4_weight &w, const uint16_t *x, int m,
                                 uint16_t *y, void *ws, const DeviceInfo &dev,
                                 cudaStream_t st);

size_t step_plan_bytes(int n_proj);
aq_status step_plan_create(const aq_nvfp4_weight *w, int n_proj, const uint16_t *const *x,
                           uint16_t *const *y, int m, void *plan, size_t plan_bytes,
                           size_t *ws_bytes, const DeviceInfo &dev);
cudaError_t launch_step(const void *plan, int m, void *ws, size_t ws_bytes, const DeviceInfo &dev,
                        cudaStream_t st);

}  // namespace aq

// Host-only checks of one GEMV call's arguments (api.cu).
extern "C" aq_status gemv_args(const aq_nvfp4_weight *w, const uint16_t *x, int32_t m, const uint16_t *y,
                    aq_path path, const char *what);
