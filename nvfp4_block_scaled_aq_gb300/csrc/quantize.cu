// quantize.cu -- load-time kernels: theta reconstruction, per-tensor amax
// and round-to-nearest NVFP4 quantisation (plain, or fused with the
// reconstruction so W_eff never reaches memory), plus the scale-layout
// unswizzle used by tests.
//
// Method: AttnQuant docs, landing page "How it works" (W_eff = s*W0 +
// U*V^T, rebuilt once at load) and "Results" (round-to-nearest, no
// calibration); "GPU acceleration", "NVFP4 quantization" (packed uint8
// nibbles + float8 block scales); "Throughput", "What quantization
// actually saves" (one float8_e4m3fn scale per 16 elements).
//
// Every fp32 step that decides a stored bit uses an explicitly rounded
// intrinsic (__fmul_rn, __fdiv_rn, __fmaf_rn) so the compiler cannot fuse
// or reorder it.
#include "aq_internal.cuh"

namespace aq {
namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------- reconstruction

// One element of W_eff in fp32 (before the bf16 rounding): the rank term
// first (fma chain from +0, t ascending), then s*w0 alone if the rank term
// is zero, else one fma.
template <int R>
__device__ __forceinline__ float recon_elem(float w0, float s, const float *u,
                                            const uint16_t *vrow, int r) {
  float delta = 0.0f;
  if (R == 4) {
    // the row's four bf16 in one 8-byte load (V is 8-byte aligned whenever
    // this instantiation is launched)
    const uint2 vv = __ldg(reinterpret_cast<const uint2 *>(vrow));
    delta = __fmaf_rn(u[0], bf16_lo(vv.x), delta);
    delta = __fmaf_rn(u[1], bf16_hi(vv.x), delta);
    delta = __fmaf_rn(u[2], bf16_lo(vv.y), delta);
    delta = __fmaf_rn(u[3], bf16_hi(vv.y), delta);
  } else if (R >= 0) {
#pragma unroll
    for (int t = 0; t < R; ++t)
      delta = __fmaf_rn(u[t], __uint_as_float(uint32_t(vrow[t]) << 16), delta);
  } else {
    for (int t = 0; t < r; ++t)
      delta = __fmaf_rn(u[t], __uint_as_float(uint32_t(__ldg(vrow + t)) << 16), delta);
  }
  return delta == 0.0f ? __fmul_rn(s, w0) : __fmaf_rn(s, w0, delta);
}

// Up to 64 rank entries of one U row, as fp32.
template <int R>
__device__ __forceinline__ void load_urow(float *u, const uint16_t *U, int64_t row,
                                          int r) {
  const int rr = R >= 0 ? R : r;
#pragma unroll
  for (int t = 0; t < (R >= 0 ? R : 64); ++t)
    if (t < rr) u[t] = __uint_as_float(uint32_t(__ldg(U + row * rr + t)) << 16);
}

template <int R>
__global__ void __launch_bounds__(kThreads)
    reconstruct_kernel(const uint16_t *__restrict__ W0, const float *__restrict__ s,
                       const uint16_t *__restrict__ U, const uint16_t *__restrict__ V,
                       int n, int k, int r, uint16_t *__restrict__ W_eff) {
  const int64_t per_row = k / 8;
  const int64_t total = int64_t(n) * per_row;
  float u[R >= 0 ? (R > 0 ? R : 1) : 64];
  for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = idx / per_row;
    const int64_t col = (idx - row * per_row) * 8;
    const uint4 wv = *reinterpret_cast<const uint4 *>(W0 + row * k + col);
    const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
    const float srow = __ldg(s + row);
    if (R != 0) load_urow<R>(u, U, row, r);
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int rr = R >= 0 ? R : r;
      float lo = recon_elem<R>(bf16_lo(w[i]), srow, u, V + (col + 2 * i) * rr, r);
      float hi = recon_elem<R>(bf16_hi(w[i]), srow, u, V + (col + 2 * i + 1) * rr, r);
      out[i] = uint32_t(f32_to_bf16_rn(lo)) | (uint32_t(f32_to_bf16_rn(hi)) << 16);
    }
    *reinterpret_cast<uint4 *>(W_eff + row * k + col) =
        make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// ---------------------------------------------------------- amax
// max |w| is taken on bf16 bit patterns with the sign cleared: for
// non-negative values the integer order is the value order, and NaN / inf
// patterns sort above every finite value, so a non-finite tensor shows up
// as amax >= 0x7F80.

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v) {
  __shared__ uint32_t red[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  v = 0;
  if (threadIdx.x < kThreads / 32) v = red[threadIdx.x];
  if (threadIdx.x < 32) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  }
  return v;
}

__global__ void __launch_bounds__(kThreads)
    amax_kernel(const uint16_t *__restrict__ W, int64_t count8, uint32_t *amax_bits) {
  uint32_t m2 = 0;  // two u16 maxima side by side
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < count8;
       i += int64_t(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(W) + i);
    m2 = __vmaxu2(m2, v.x & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v.y & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v.w & 0x7FFF7FFFu);
  }
  uint32_t m = block_max_u32(max(m2 & 0xFFFFu, m2 >> 16));
  if (threadIdx.x == 0) atomicMax(amax_bits, m);
}

template <int R>
__global__ void __launch_bounds__(kThreads)
    amax_fused_kernel(const uint16_t *__restrict__ W0, const float *__restrict__ s,
                      const uint16_t *__restrict__ U, const uint16_t *__restrict__ V,
                      int n, int k, int r, uint32_t *amax_bits) {
  const int64_t per_row = k / 8;
  const int64_t total = int64_t(n) * per_row;
  float u[R >= 0 ? (R > 0 ? R : 1) : 64];
  uint32_t m = 0;
  for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = idx / per_row;
    const int64_t col = (idx - row * per_row) * 8;
    const uint4 wv = __ldg(reinterpret_cast<const uint4 *>(W0 + row * k + col));
    const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
    const float srow = __ldg(s + row);
    if (R != 0) load_urow<R>(u, U, row, r);
    const int rr = R >= 0 ? R : r;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float lo = recon_elem<R>(bf16_lo(w[i]), srow, u, V + (col + 2 * i) * rr, r);
      float hi = recon_elem<R>(bf16_hi(w[i]), srow, u, V + (col + 2 * i + 1) * rr, r);
      m = max(m, uint32_t(f32_to_bf16_rn(lo)) & 0x7FFFu);
      m = max(m, uint32_t(f32_to_bf16_rn(hi)) & 0x7FFFu);
    }
  }
  m = block_max_u32(m);
  if (threadIdx.x == 0) atomicMax(amax_bits, m);
}

// ---------------------------------------------------------- quantise

// Per-tensor scales from the amax bits; false if amax is out of range.
__device__ __forceinline__ bool global_scales(uint32_t amax_bits, float &g_enc,
                                              float &g_dec) {
  if (amax_bits >= 0x7F80u) return false;  // inf or NaN
  const float a = __uint_as_float(amax_bits << 16);
  if (a == 0.0f) {
    g_enc = 1.0f;
    g_dec = 1.0f;
    return true;
  }
  g_enc = __fdiv_rn(kGlobalMax, a);
  g_dec = __fdiv_rn(a, kGlobalMax);
  return !isinf(g_enc);
}

// Quantise one 16-element block held as fp32 in w[0..15]: returns the E4M3
// scale code and writes 8 packed bytes as two 32-bit words.
__device__ __forceinline__ uint32_t quantize_block(const float *w, float g_enc,
                                                   uint32_t &lo, uint32_t &hi) {
  float b = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) b = fmaxf(b, fabsf(w[i]));
  const float t = __fmul_rn(__fdiv_rn(b, 6.0f), g_enc);
  const uint32_t sf = f32x2_to_e4m3x2(0.0f, t) & 0xFFu;
  const uint32_t sd_h2 = e4m3x2_to_f16x2(uint16_t(sf));
  const float sd = f16_lo_to_f32(sd_h2);
  lo = hi = 0;
  if (sd != 0.0f) {
    const float rcp = __fdiv_rn(g_enc, sd);
    uint32_t bytes[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float v0 = __fmul_rn(w[2 * i], rcp);
      const float v1 = __fmul_rn(w[2 * i + 1], rcp);
      // the conversion keeps the sign, a negative value that rounds to zero
      // included (nibble 0x8); the sweep over every bf16 value checks it
      bytes[i] = f32x2_to_e2m1x2(v1, v0);
    }
    lo = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24);
    hi = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (bytes[7] << 24);
  }
  return sf;
}

// One warp per 16 x 128 tile; lane 4g + c owns rows g and g + 8 of the
// tile and columns [32c, 32c + 32), i.e. two blocks per row, and writes the
// one 32-bit scale word of the layout that holds exactly those four scales.
template <int R, bool kFused>
__global__ void __launch_bounds__(kThreads)
    quantize_kernel(const uint16_t *__restrict__ W, const float *__restrict__ s,
                    const uint16_t *__restrict__ U, const uint16_t *__restrict__ V,
                    int n, int k, int r, uint8_t *__restrict__ packed,
                    uint8_t *__restrict__ scales, float *__restrict__ global_scale,
                    const uint32_t *__restrict__ amax_bits, unsigned *status) {
  float g_enc = 1.0f, g_dec = 1.0f;
  const bool ok = global_scales(*amax_bits, g_enc, g_dec);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *global_scale = ok ? g_dec : __int_as_float(0x7FC00000);
    if (!ok) raise_status(status, kDevRange);
  }
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t tiles_k = ceil_div(k, kTileCols);
  const int64_t tiles = ceil_div(n, kTileRows) * tiles_k;
  const int64_t warp0 = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  float u[R >= 0 ? (R > 0 ? R : 1) : 64];
  for (int64_t tile = warp0; tile < tiles; tile += nwarps) {
    const int64_t tn = tile / tiles_k, tk = tile - tn * tiles_k;
    const int64_t col = tk * kTileCols + 32 * c;
    uint32_t sword = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t row = tn * kTileRows + 8 * h + g;
      if (row >= n || col >= k) continue;
      float w[32];
      if (!kFused) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = __ldg(reinterpret_cast<const uint4 *>(W + row * k + col) + q);
          const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            w[8 * q + 2 * i] = bf16_lo(vv[i]);
            w[8 * q + 2 * i + 1] = bf16_hi(vv[i]);
          }
        }
      } else {
        const float srow = __ldg(s + row);
        if (R != 0) load_urow<R>(u, U, row, r);
        const int rr = R >= 0 ? R : r;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = __ldg(reinterpret_cast<const uint4 *>(W + row * k + col) + q);
          const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int64_t j = col + 8 * q + 2 * i;
            const float lo = recon_elem<R>(bf16_lo(vv[i]), srow, u, V + j * rr, r);
            const float hi = recon_elem<R>(bf16_hi(vv[i]), srow, u, V + (j + 1) * rr, r);
            w[8 * q + 2 * i] = __uint_as_float(uint32_t(f32_to_bf16_rn(lo)) << 16);
            w[8 * q + 2 * i + 1] = __uint_as_float(uint32_t(f32_to_bf16_rn(hi)) << 16);
          }
        }
      }
      uint4 out = make_uint4(0, 0, 0, 0);
      uint32_t sf0 = 0, sf1 = 0;
      if (ok) {
        sf0 = quantize_block(w, g_enc, out.x, out.y);
        sf1 = quantize_block(w + 16, g_enc, out.z, out.w);
      }
      *reinterpret_cast<uint4 *>(packed + row * (k / 2) + col / 2) = out;
      sword |= (sf0 | (sf1 << 8)) << (16 * h);
    }
    reinterpret_cast<uint32_t *>(scales + tile * 128)[lane] = sword;
  }
}

// ---------------------------------------------------------- rank 4, V reused
// The fused form for the configured rank (4) with V 16-byte aligned.  Each
// warp keeps one 128-column tile column for its whole life and walks down
// its row tiles (warps w and w + P * tiles_k share a tile column; P row
// tiles are in flight per column), so the V rows it reads stay in L1; per
// 16-column block lane (g, c) loads the block's V rows once (128 bytes,
// eight 16-byte loads) and rebuilds rows g and g + 8 from them.  The
// arithmetic is recon_elem<4>'s, in the same order.

// One element of the rank-4 rebuild (fp32, before the bf16 rounding) from V
// values already in registers: recon_elem<4>'s value.  The zero-delta case
// (s * w0 alone) is one fma with -0 as the addend: fma(s, w0, -0) is the
// product rounded once, -0 when the product is -0 and +0 when it is +0,
// exactly as the rounded product itself.
__device__ __forceinline__ float recon4(float w0, float s, const float (&u)[4], uint32_t v01,
                                        uint32_t v23) {
  float delta = 0.0f;
  delta = __fmaf_rn(u[0], bf16_lo(v01), delta);
  delta = __fmaf_rn(u[1], bf16_hi(v01), delta);
  delta = __fmaf_rn(u[2], bf16_lo(v23), delta);
  delta = __fmaf_rn(u[3], bf16_hi(v23), delta);
  return __fmaf_rn(s, w0, delta == 0.0f ? -0.0f : delta);
}

// Two fp32 -> bf16x2 (nearest even), `hi` in the upper half.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float hi, float lo) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// V rows of the 16 columns starting at col: column j's four entries in
// vr[2j] (entries 0, 1) and vr[2j + 1] (entries 2, 3).
__device__ __forceinline__ void load_v16(const uint16_t *__restrict__ V, int64_t col,
                                         uint32_t (&vr)[32]) {
  const uint4 *src = reinterpret_cast<const uint4 *>(V + col * 4);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 v = __ldg(src + i);
    vr[4 * i] = v.x;
    vr[4 * i + 1] = v.y;
    vr[4 * i + 2] = v.z;
    vr[4 * i + 3] = v.w;
  }
}

// The 16 rebuilt values (bf16-rounded, as fp32) of row `row`, columns
// col .. col + 15.
__device__ __forceinline__ void rebuild16(const uint16_t *__restrict__ W0, float srow,
                                          const float (&u)[4], int k, int64_t row, int64_t col,
                                          const uint32_t (&vr)[32], float (&w)[16]) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(W0 + row * k + col) + q);
    const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = 8 * q + 2 * i;
      const float lo = recon4(bf16_lo(vv[i]), srow, u, vr[2 * j], vr[2 * j + 1]);
      const float hi = recon4(bf16_hi(vv[i]), srow, u, vr[2 * j + 2], vr[2 * j + 3]);
      const uint32_t b2 = f32x2_to_bf16x2(hi, lo);
      w[j] = bf16_lo(b2);
      w[j + 1] = bf16_hi(b2);
    }
  }
}

// max over the 16 values of |e| (fp32, before the bf16 rounding) as bit
// patterns with the sign cleared, so a NaN or an infinity sorts above every
// finite value.  Rounding to nearest is monotonic in magnitude, so the
// largest |bf16(e)| is bf16 of the largest |e|: the caller rounds once.
__device__ __forceinline__ uint32_t rebuild16_absmax(const uint16_t *__restrict__ W0, float srow,
                                                     const float (&u)[4], int k, int64_t row,
                                                     int64_t col, const uint32_t (&vr)[32],
                                                     uint32_t m) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(W0 + row * k + col) + q);
    const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = 8 * q + 2 * i;
      const float lo = recon4(bf16_lo(vv[i]), srow, u, vr[2 * j], vr[2 * j + 1]);
      const float hi = recon4(bf16_hi(vv[i]), srow, u, vr[2 * j + 2], vr[2 * j + 3]);
      m = max(m, __float_as_uint(lo) & 0x7FFFFFFFu);
      m = max(m, __float_as_uint(hi) & 0x7FFFFFFFu);
    }
  }
  return m;
}

__device__ __forceinline__ void row_terms(const float *__restrict__ s,
                                          const uint16_t *__restrict__ U, int64_t row,
                                          float &srow, float (&u)[4]) {
  srow = __ldg(s + row);
#pragma unroll
  for (int t = 0; t < 4; ++t) u[t] = __uint_as_float(uint32_t(__ldg(U + row * 4 + t)) << 16);
}

__global__ void __launch_bounds__(kThreads)
    amax_r4_kernel(const uint16_t *__restrict__ W0, const float *__restrict__ s,
                   const uint16_t *__restrict__ U, const uint16_t *__restrict__ V, int n,
                   int k, int rows_in_flight, uint32_t *amax_bits) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t tiles_k = ceil_div(k, kTileCols), tiles_n = ceil_div(n, kTileRows);
  const int64_t warp = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5;
  uint32_t m = 0;
  if (warp < tiles_k * rows_in_flight) {
    const int64_t tk = warp % tiles_k, tn0 = warp / tiles_k;
    const int64_t col = tk * kTileCols + 32 * c;
    if (col < k)
      for (int64_t tn = tn0; tn < tiles_n; tn += rows_in_flight) {
        float srow[2], u[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t row = tn * kTileRows + 8 * h + g;
          if (row < n) row_terms(s, U, row, srow[h], u[h]);
        }
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          uint32_t vr[32];
          load_v16(V, col + 16 * b, vr);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int64_t row = tn * kTileRows + 8 * h + g;
            if (row >= n) continue;
            m = rebuild16_absmax(W0, srow[h], u[h], k, row, col + 16 * b, vr, m);
          }
        }
      }
  }
  // bf16 bits of the largest |e|: a NaN stays a NaN pattern and an
  // infinity the infinity pattern, both at or above 0x7F80
  uint32_t mb = m >= 0x7F800000u ? (m >> 16) | (m > 0x7F800000u ? 0x40u : 0u)
                                 : uint32_t(f32_to_bf16_rn(__uint_as_float(m)));
  mb = block_max_u32(mb);
  if (threadIdx.x == 0) atomicMax(amax_bits, mb);
}

__global__ void __launch_bounds__(kThreads)
    quantize_r4_kernel(const uint16_t *__restrict__ W0, const float *__restrict__ s,
                       const uint16_t *__restrict__ U, const uint16_t *__restrict__ V, int n,
                       int k, int rows_in_flight, uint8_t *__restrict__ packed,
                       uint8_t *__restrict__ scales, float *__restrict__ global_scale,
                       const uint32_t *__restrict__ amax_bits, unsigned *status) {
  float g_enc = 1.0f, g_dec = 1.0f;
  const bool ok = global_scales(*amax_bits, g_enc, g_dec);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *global_scale = ok ? g_dec : __int_as_float(0x7FC00000);
    if (!ok) raise_status(status, kDevRange);
  }
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t tiles_k = ceil_div(k, kTileCols), tiles_n = ceil_div(n, kTileRows);
  const int64_t warp = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5;
  if (warp >= tiles_k * rows_in_flight) return;
  const int64_t tk = warp % tiles_k, tn0 = warp / tiles_k;
  const int64_t col = tk * kTileCols + 32 * c;
  for (int64_t tn = tn0; tn < tiles_n; tn += rows_in_flight) {
    float srow[2], u[2][4];
    uint32_t out[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
    uint32_t sword = 0;
    if (col < k) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t row = tn * kTileRows + 8 * h + g;
        if (row < n) row_terms(s, U, row, srow[h], u[h]);
      }
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        uint32_t vr[32];
        load_v16(V, col + 16 * b, vr);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t row = tn * kTileRows + 8 * h + g;
          if (row >= n) continue;
          float w[16];
          rebuild16(W0, srow[h], u[h], k, row, col + 16 * b, vr, w);
          uint32_t sf = 0;
          if (ok) sf = quantize_block(w, g_enc, out[h][2 * b], out[h][2 * b + 1]);
          sword |= sf << (16 * h + 8 * b);
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t row = tn * kTileRows + 8 * h + g;
        if (row < n)
          *reinterpret_cast<uint4 *>(packed + row * (k / 2) + col / 2) =
              make_uint4(out[h][0], out[h][1], out[h][2], out[h][3]);
      }
    }
    reinterpret_cast<uint32_t *>(scales + (tn * tiles_k + tk) * 128)[lane] = sword;
  }
}

// Activations for the block-scaled MMA path (reading R9: each token row
// quantised on its own, with the per-tensor steps applied per row): one CTA
// per row.  packed [m, k/2], scales [m, k/16] row-major with a row pitch of
// scale_pitch bytes (k/16 for the canonical layout), g_dec [m].  A row whose amax is out of range is zero-filled, gets a NaN
// g_dec and raises AQ_ERR_RANGE.
__global__ void __launch_bounds__(kThreads)
    act_quant_kernel(const uint16_t *__restrict__ x, int k, uint8_t *__restrict__ packed,
                     uint8_t *__restrict__ scales, int scale_pitch, float *__restrict__ g_dec,
                     unsigned *status) {
  __shared__ uint32_t amax_s;
  const int64_t row = blockIdx.x;
  const uint16_t *xr = x + row * k;
  uint32_t m2 = 0;
  for (int i = threadIdx.x * 8; i < k; i += kThreads * 8) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xr + i));
    m2 = __vmaxu2(m2, v.x & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v.y & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v.w & 0x7FFF7FFFu);
  }
  const uint32_t m = block_max_u32(max(m2 & 0xFFFFu, m2 >> 16));
  if (threadIdx.x == 0) amax_s = m;
  __syncthreads();
  float g_enc = 1.0f, gd = 1.0f;
  const bool ok = global_scales(amax_s, g_enc, gd);
  if (threadIdx.x == 0) {
    g_dec[row] = ok ? gd : __int_as_float(0x7FC00000);
    if (!ok) raise_status(status, kDevRange);
  }
  for (int b = threadIdx.x; b < k / kBlock; b += kThreads) {
    float w[16];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xr + b * kBlock) + q);
      const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        w[8 * q + 2 * i] = bf16_lo(vv[i]);
        w[8 * q + 2 * i + 1] = bf16_hi(vv[i]);
      }
    }
    uint32_t lo = 0, hi = 0, sf = 0;
    if (ok) sf = quantize_block(w, g_enc, lo, hi);
    *reinterpret_cast<uint2 *>(packed + row * (k / 2) + b * 8) = make_uint2(lo, hi);
    scales[row * scale_pitch + b] = uint8_t(sf);
  }
}

__global__ void scales_to_canonical_kernel(const uint8_t *__restrict__ scales, int n,
                                           int k, uint8_t *__restrict__ canon) {
  const int64_t nblk = k / kBlock;
  const int64_t total = int64_t(n) * nblk;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = i / nblk, blk = i - row * nblk;
    canon[i] = scales[scale_offset(row, blk, k)];
  }
}

int grid_for(int64_t work, int per_cta, int cap) {
  int64_t g = ceil_div(work, per_cta);
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return int(g);
}

}  // namespace

cudaError_t launch_reconstruct(const uint16_t *W0, const float *s, const uint16_t *U,
                               const uint16_t *V, int n, int k, int r, uint16_t *W_eff,
                               cudaStream_t st) {
  const int grid = grid_for(int64_t(n) * (k / 8), kThreads, 152 * 16);
  if (r == 0)
    reconstruct_kernel<0><<<grid, kThreads, 0, st>>>(W0, s, U, V, n, k, r, W_eff);
  else if (r == 4 && (reinterpret_cast<uintptr_t>(V) & 7u) == 0)
    reconstruct_kernel<4><<<grid, kThreads, 0, st>>>(W0, s, U, V, n, k, r, W_eff);
  else
    reconstruct_kernel<-1><<<grid, kThreads, 0, st>>>(W0, s, U, V, n, k, r, W_eff);
  return cudaGetLastError();
}

template <int R, bool kFused>
static void quantize_pass(const uint16_t *W, const float *s, const uint16_t *U,
                          const uint16_t *V, int r, int n, int k,
                          const aq_nvfp4_weight &out, uint32_t *amax, const DeviceInfo &dev,
                          cudaStream_t st) {
  const int cap = dev.sms * 8;
  if (kFused) {
    const int g = grid_for(int64_t(n) * (k / 8), kThreads, cap);
    amax_fused_kernel<R><<<g, kThreads, 0, st>>>(W, s, U, V, n, k, r, amax);
  } else {
    const int g = grid_for(int64_t(n) * k / 8, kThreads, cap);
    amax_kernel<<<g, kThreads, 0, st>>>(W, int64_t(n) * k / 8, amax);
  }
  const int64_t tiles = ceil_div(n, kTileRows) * ceil_div(k, kTileCols);
  const int g = grid_for(tiles, kThreads / 32, cap);
  quantize_kernel<R, kFused><<<g, kThreads, 0, st>>>(W, s, U, V, n, k, r, out.packed,
                                                     out.scales, out.global_scale, amax,
                                                     dev.status);
}

// Rank 4 with V reused per warp: P row tiles in flight per tile column,
// about sixteen warps per SM in all (two CTAs of eight, one wave).
static void quantize_pass_r4(const uint16_t *W, const float *s, const uint16_t *U,
                             const uint16_t *V, int n, int k, const aq_nvfp4_weight &out,
                             uint32_t *amax, const DeviceInfo &dev, cudaStream_t st) {
  const int64_t tiles_k = ceil_div(k, kTileCols), tiles_n = ceil_div(n, kTileRows);
  int64_t P = int64_t(dev.sms) * 16 / tiles_k;
  if (P < 1) P = 1;
  if (P > tiles_n) P = tiles_n;
  const int warps_per_cta = kThreads / 32;
  const int g = int(ceil_div(tiles_k * P, warps_per_cta));
  amax_r4_kernel<<<g, kThreads, 0, st>>>(W, s, U, V, n, k, int(P), amax);
  quantize_r4_kernel<<<g, kThreads, 0, st>>>(W, s, U, V, n, k, int(P), out.packed, out.scales,
                                             out.global_scale, amax, dev.status);
}

cudaError_t launch_quantize(const uint16_t *W, const float *s, const uint16_t *U,
                            const uint16_t *V, int r, bool fused, int n, int k,
                            const aq_nvfp4_weight &out, void *ws, const DeviceInfo &dev,
                            cudaStream_t st) {
  uint32_t *amax = static_cast<uint32_t *>(ws);
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  if (!fused)
    quantize_pass<0, false>(W, s, U, V, 0, n, k, out, amax, dev, st);
  else if (r == 4 && (reinterpret_cast<uintptr_t>(V) & 15u) == 0)
    quantize_pass_r4(W, s, U, V, n, k, out, amax, dev, st);
  else if (r == 0)
    quantize_pass<0, true>(W, s, U, V, r, n, k, out, amax, dev, st);
  else if (r == 4 && (reinterpret_cast<uintptr_t>(V) & 7u) == 0)
    quantize_pass<4, true>(W, s, U, V, r, n, k, out, amax, dev, st);
  else
    quantize_pass<-1, true>(W, s, U, V, r, n, k, out, amax, dev, st);
  return cudaGetLastError();
}

cudaError_t launch_act_quant(const uint16_t *x, int m, int k, uint8_t *packed, uint8_t *scales,
                             int scale_pitch, float *g_dec, const DeviceInfo &dev,
                             cudaStream_t st) {
  act_quant_kernel<<<m, kThreads, 0, st>>>(x, k, packed, scales, scale_pitch, g_dec, dev.status);
  return cudaGetLastError();
}

// out row 16 j + i = gate row 8 j + i, out row 16 j + 8 + i = up row 8 j + i
// (i < 8) of the row-concatenated [gate; up] weight w [2f, k]: one 16-byte
// vector per thread, grid-stride.
__global__ void interleave_gate_up_kernel(const uint4 *__restrict__ w, int f, int k,
                                          uint4 *__restrict__ out) {
  const int64_t vpr = k / 8;  // 16-byte vectors per row
  const int64_t total = int64_t(2) * f * vpr;
  for (int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; v < total;
       v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = v / vpr, col = v - row * vpr;
    const int64_t grp = row / 16, within = row % 16;
    const int64_t src = within < 8 ? grp * 8 + within : f + grp * 8 + (within - 8);
    out[v] = w[src * vpr + col];
  }
}

cudaError_t launch_interleave_gate_up(const uint16_t *w, int f, int k, uint16_t *out,
                                      cudaStream_t st) {
  const int grid = grid_for(int64_t(2) * f * (k / 8), 256, 152 * 16);
  interleave_gate_up_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const uint4 *>(w), f, k,
                                                  reinterpret_cast<uint4 *>(out));
  return cudaGetLastError();
}

cudaError_t launch_scales_to_canonical(const aq_nvfp4_weight &w, uint8_t *canon,
                                       cudaStream_t st) {
  const int grid = grid_for(int64_t(w.n) * (w.k / kBlock), 256, 152 * 8);
  scales_to_canonical_kernel<<<grid, 256, 0, st>>>(w.scales, w.n, w.k, canon);
  return cudaGetLastError();
}

}  // namespace aq
