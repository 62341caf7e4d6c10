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
#include <cstring>
#include <mutex>

#include "aq_internal.cuh"
#include "gemv_core.cuh"

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

template <int kBlockThreads = kThreads>
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v) {
  __shared__ uint32_t red[kBlockThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  v = 0;
  if (threadIdx.x < kBlockThreads / 32) v = red[threadIdx.x];
  if (threadIdx.x < 32) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  }
  return v;
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

// Called by every thread of a CTA after a __syncthreads that follows all of
// its threads' reads of the amax word: the CTA counts itself out on
// ws[2], and the last CTA of the grid clears ws[0..2] (amax, grid
// arrivals, departures), so the call leaves the workspace zeroed.
__device__ __forceinline__ void depart_and_clear(uint32_t *ws) {
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(ws + 2, 1u) == gridDim.x - 1) {
      ws[0] = 0;
      ws[1] = 0;
      ws[2] = 0;
      __threadfence();
    }
  }
}

// Two fp32 -> bf16x2 (nearest even), `hi` in the upper half.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float hi, float lo) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// The bf16 pair w (element 0 in the low half) as an fp32 pair.
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
  return pack2(bf16_lo(w), bf16_hi(w));
}

// RN(b / 6) for a non-negative bf16 value b held as fp32: the product with
// RN(1/6), corrected by one fma residual step.  For every such b (+0, the
// subnormals, every finite normal; verified exhaustively) this is the
// correctly rounded quotient, __fdiv_rn(b, 6.0f).
__device__ __forceinline__ float div6_rn(float b) {
  const float c = 0x1.555556p-3f;  // 1/6 rounded to nearest
  const float q0 = __fmul_rn(b, c);
  return __fmaf_rn(__fmaf_rn(-6.0f, q0, b), c, q0);
}

// rcp_tab[code] = RN(g_enc / decode(code)) for the E4M3 codes a block scale
// can take (1 .. 0x7E; entry 0 unused).  The caller synchronises before the
// first read.
__device__ __forceinline__ void fill_rcp_table(float g_enc, float *rcp_tab) {
  for (int i = threadIdx.x; i < 128; i += blockDim.x) {
    const float sd = f16_lo_to_f32(e4m3x2_to_f16x2(uint16_t(i)));
    rcp_tab[i] = i == 0 ? 0.0f : __fdiv_rn(g_enc, sd);
  }
}

// Eight bf16 values (pairs w0 .. w3, element 2i in the low half of word i)
// times rcp, each product rounded to fp32 and converted to E2M1 (nearest
// even, saturated at 6, sign kept, also for a magnitude that rounds to
// zero): one 32-bit word, element 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t e2m1x8_scaled(uint32_t w0, uint32_t w1, uint32_t w2,
                                                  uint32_t w3, uint64_t r2) {
  const uint32_t w[4] = {w0, w1, w2, w3};
  float p[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint64_t v;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(v) : "l"(bf16x2_to_f32x2(w[i])), "l"(r2));
    unpack2(v, p[2 * i], p[2 * i + 1]);
  }
  uint32_t out;
  asm("{ .reg .b8 b0, b1, b2, b3;\n"
      "  cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      "  cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      "  cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      "  cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      "  mov.b32 %0, {b0, b1, b2, b3}; }"
      : "=r"(out)
      : "f"(p[0]), "f"(p[1]), "f"(p[2]), "f"(p[3]), "f"(p[4]), "f"(p[5]), "f"(p[6]),
        "f"(p[7]));
  return out;
}

// Quantise one 16-element block given as eight bf16 pairs (element 2i in
// the low half of bw[i]): returns the E4M3 scale code and writes the eight
// packed bytes as two 32-bit words.  b = max |w| is the larger magnitude of
// a max.xorsign.abs chain over the pairs (the sign it leaves is dropped);
// sf = E4M3(RN(RN(b / 6) * g_enc)); if sf decodes to 0 (code 0) the nibbles
// are 0, else nibble i = E2M1(RN(w_i * rcp_tab[sf])).
__device__ __forceinline__ uint32_t quantize_block16(const uint32_t (&bw)[8], float g_enc,
                                                     const float *__restrict__ rcp_tab,
                                                     uint32_t &lo, uint32_t &hi) {
  uint32_t m = bw[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(bw[i]));
  const uint32_t bb = max(m & 0x7FFFu, (m >> 16) & 0x7FFFu);
  const float t = __fmul_rn(div6_rn(__uint_as_float(bb << 16)), g_enc);
  const uint32_t sf = f32x2_to_e4m3x2(0.0f, t) & 0xFFu;
  lo = hi = 0;
  if (sf != 0) {
    const float rcp = rcp_tab[sf];
    const uint64_t r2 = pack2(rcp, rcp);
    lo = e2m1x8_scaled(bw[0], bw[1], bw[2], bw[3], r2);
    hi = e2m1x8_scaled(bw[4], bw[5], bw[6], bw[7], r2);
  }
  return sf;
}

// The fused form for ranks and alignments the rank-4 kernel does not serve:
// one warp per 16 x 128 tile; lane 4g + c owns rows g and g + 8 of the tile
// and columns [32c, 32c + 32), i.e. two blocks per row, and writes the one
// 32-bit scale word of the layout that holds exactly those four scales.
template <int R>
__global__ void __launch_bounds__(kThreads)
    quantize_kernel(const uint16_t *__restrict__ W, const float *__restrict__ s,
                    const uint16_t *__restrict__ U, const uint16_t *__restrict__ V,
                    int n, int k, int r, uint8_t *__restrict__ packed,
                    uint8_t *__restrict__ scales, float *__restrict__ global_scale,
                    uint32_t *amax_bits, unsigned *status) {
  float g_enc = 1.0f, g_dec = 1.0f;
  const bool ok = global_scales(*amax_bits, g_enc, g_dec);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *global_scale = ok ? g_dec : __int_as_float(0x7FC00000);
    if (!ok) raise_status(status, kDevRange);
  }
  __shared__ float rcp_tab[128];
  fill_rcp_table(g_enc, rcp_tab);
  __syncthreads();
  depart_and_clear(amax_bits);
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
      uint32_t bw[2][8];  // the row's 32 values as bf16 pairs, per block
      {
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
            bw[q >> 1][4 * (q & 1) + i] = f32x2_to_bf16x2(hi, lo);
          }
        }
      }
      uint4 out = make_uint4(0, 0, 0, 0);
      uint32_t sf0 = 0, sf1 = 0;
      if (ok) {
        sf0 = quantize_block16(bw[0], g_enc, rcp_tab, out.x, out.y);
        sf1 = quantize_block16(bw[1], g_enc, rcp_tab, out.z, out.w);
      }
      *reinterpret_cast<uint4 *>(packed + row * (k / 2) + col / 2) = out;
      sword |= (sf0 | (sf1 << 8)) << (16 * h);
    }
    reinterpret_cast<uint32_t *>(scales + tile * 128)[lane] = sword;
  }
}

// ---------------------------------------------------------- rank 4, packed fp32
// The fused form for the configured rank (4) with V, U and s 16-byte
// aligned.  Warp w of W works tile column w % tiles_k, whose W_c warps
// (W / tiles_k, one more for the first W % tiles_k columns) take its row
// tiles in turn; the eight warps of a CTA hold neighbouring tile columns, so
// a CTA reads 16-row bands of up to 2 KB per row.  Lane 4g + c owns rows g
// and g + 8 of each tile and columns [32c, 32c + 32): two 16-element blocks
// per row, whose four E4M3 scales form the lane's word of the scale layout.
//
// The warp's 128 columns of V sit in shared memory as fp32, rank-major
// (vt[t][c][j] = V[col0 + 32c + j][t]), so one 16-byte shared load gives
// rank entry t of four consecutive columns: two (column j, column j + 1)
// pairs for the packed fp32 fma, which rebuilds two neighbouring elements of
// a row per instruction.  Each chunk row is padded to 36 floats so that the
// four chunks' loads fall in different banks.
//
// Arithmetic, element by element the operations of recon_elem<4>: the rank
// term is an fma chain over t ascending from +0, run here on -u (an exact
// negation), so it ends at m = -delta when delta != 0 and at m = +0 when
// delta == 0 (round-to-nearest gives a zero sum the sign -0 only when both
// addends are -0, and the chain starts at +0).  fma(s, w0, -m) is then
// fma(s, w0, delta) when delta != 0, exact cancellation included, and
// fma(s, w0, -0) = s * w0 rounded once, with the product's own sign of
// zero, when delta == 0.  The amax pass needs only |e|, which the sign of a
// zero does not change, so it takes fma(-s, w0, m) = -e on packed pairs.
// The quantisation pass walks its row tiles in the reverse order, so that it
// starts on the weights the amax pass read last, while they are still in L2.

constexpr int kVtPitch = 36;                 // floats per (rank, chunk) row
constexpr int kVtFloats = 4 * 4 * kVtPitch;  // one warp's V tile

// Element-wise a * b + c on fp32 pairs, each rounded once (fma.rn.f32).
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Stage the warp's V tile, negated (-v is exact, and fma(u, -v, m)
// equals fma(-u, v, m)): lane l converts columns col0 + 4l .. + 3 (two
// 16-byte loads of four bf16 rank entries per column); columns at or past k
// are zero.
__device__ __forceinline__ void stage_vt(const uint16_t *__restrict__ V, int64_t col0, int k,
                                         int lane, float *vt) {
  const int64_t cb = col0 + 4 * lane;
  uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
  if (cb < k) {
    a = __ldg(reinterpret_cast<const uint4 *>(V + cb * 4));
    b = __ldg(reinterpret_cast<const uint4 *>(V + cb * 4) + 1);
  }
  // column cb + q, rank t: word (2q + t / 2) of (a, b), half t % 2
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  const int ch = lane >> 3, j = 4 * (lane & 7);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    float4 v;
    v.x = -((t & 1) ? bf16_hi(w[0 + (t >> 1)]) : bf16_lo(w[0 + (t >> 1)]));
    v.y = -((t & 1) ? bf16_hi(w[2 + (t >> 1)]) : bf16_lo(w[2 + (t >> 1)]));
    v.z = -((t & 1) ? bf16_hi(w[4 + (t >> 1)]) : bf16_lo(w[4 + (t >> 1)]));
    v.w = -((t & 1) ? bf16_hi(w[6 + (t >> 1)]) : bf16_lo(w[6 + (t >> 1)]));
    *reinterpret_cast<float4 *>(vt + (t * 4 + ch) * kVtPitch + j) = v;
  }
}


// s and the U row (two bf16 pairs) of one row of a stage's tile.
struct R4Row {
  float s;
  uint32_t u01, u23;
};

// The weights reach shared memory through a two-stage ring per warp: a
// stage holds one row tile of the warp's tile column as two TMA boxes of 16
// rows x 64 columns (128 bytes per row, 128-byte swizzle: 16-byte chunk j of
// row r sits at chunk j ^ (r & 7)); rows past n and columns past k read as
// zero.  The tile's 16 U rows (128 bytes) and 16 s values (64 bytes) come
// with it, as 1-D boxes into a side buffer of the stage (zero past n).  Lane
// 0 refills a stage once every lane of the warp has read it, so two row
// tiles are in flight while the warp converts one.
constexpr int kR4Stages = 2;
constexpr int kR4BoxBytes = kTileRows * 128;    // one 16 x 64 box
constexpr int kR4StageBytes = 2 * kR4BoxBytes;  // one row tile
constexpr int kR4RowBytes = kTileRows * 8 + kTileRows * 4;  // U rows, then s
constexpr int kR4RowStride = 256;  // side buffers 128-byte aligned for the TMA

// A CTA of kWarps warps: the warps' rings, then their V tiles, their side
// buffers and their barriers.  Eight warps run as two CTAs per SM, sixteen
// as one; either way an SM holds 16 warps of up to 128 registers.  The
// rank-4 two-pass form without the hand-over runs sixteen (202 against
// 206 us on the ~31B gate+up, where two 8-warp CTAs ended between 185 and
// 204 us but every SM between 198.5 and 203); the other forms run eight, which is as fast on the ~31B
// plain quantisation and faster on the 1B shapes (16.7 against 17.5 us on
// the fused 1B down).  Ten-warp CTAs at 96 registers measured slower (219
// against 206 us).
constexpr int kR4Warps = 8, kR4WideWarps = 16;
template <int kWarps>
struct R4Geo {
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kCtasPerSm = 16 / kWarps;
  static constexpr int kRingBytes = kWarps * kR4Stages * kR4StageBytes;
  static constexpr int kRowsOffset = kRingBytes + kWarps * kVtFloats * 4;
  static constexpr int kBarsOffset = kRowsOffset + kWarps * kR4Stages * kR4RowStride;
  static constexpr int kSmemBytes = 1024 + kBarsOffset + kWarps * kR4Stages * 8;
  static_assert(kRowsOffset % 128 == 0, "TMA side buffers must be 128-byte aligned");
  static_assert(kSmemBytes <= 227 * 1024, "one CTA's shared memory");
};

struct R4Maps {
  CUtensorMap w0, u, s;
};

__device__ __forceinline__ void tma_load_1d(void *dst, const CUtensorMap *map, int x,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.1d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2}], [%3];" ::"r"(core::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(core::smem_u32(bar))
      : "memory");
}

// kPlain: a bf16 weight quantised as it is (no theta bundle): the tile's
// weights only.
template <bool kPlain>
__device__ __forceinline__ void r4_issue(const R4Maps &tm, uint8_t *stage, uint8_t *rows,
                                         uint64_t *bar, int64_t tn, int64_t col0, int k) {
  const bool two = col0 + 64 < k;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  core::mbar_expect_tx(bar, (two ? kR4StageBytes : kR4BoxBytes) + (kPlain ? 0 : kR4RowBytes));
  core::tma_load_2d(stage, &tm.w0, int(col0 * 2), int(tn * kTileRows), bar);
  if (two)
    core::tma_load_2d(stage + kR4BoxBytes, &tm.w0, int(col0 * 2 + 128), int(tn * kTileRows),
                      bar);
  if (!kPlain) {
    tma_load_1d(rows, &tm.u, int(tn * kTileRows * 8), bar);
    tma_load_1d(rows + kTileRows * 8, &tm.s, int(tn * kTileRows * 4), bar);
  }
}

__device__ __forceinline__ R4Row r4_row(const uint8_t *rows, int r) {
  const uint2 u = reinterpret_cast<const uint2 *>(rows)[r];
  return R4Row{reinterpret_cast<const float *>(rows + kTileRows * 8)[r], u.x, u.y};
}

// Lane (g, c)'s 32 columns of rows g and g + 8 from a stage: w[h][q] holds
// columns 8q .. 8q + 7 of the lane's chunk.  The four lanes of each bank
// group differ in c, so each 16-byte load takes the minimum four wavefronts.
__device__ __forceinline__ void r4_read(const uint8_t *stage, int g, int c, uint4 (&w)[2][4]) {
  const uint8_t *box = stage + (c >> 1) * kR4BoxBytes;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int q = 0; q < 4; ++q)
      w[h][q] = *reinterpret_cast<const uint4 *>(box + (8 * h + g) * 128 +
                                                 (((4 * (c & 1) + q) ^ g) << 4));
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// What r4_block does with one 16-column block of both rows:
//   kFormAmax      rebuild (packed pairs), fold |e| into mx;
//   kFormAmaxKeep  rebuild exactly (the quantisation pass's arithmetic), fold
//                  |e| into mx, and write the bf16 W_eff pairs back over the
//                  lane's W0 bytes in the stage;
//   kFormQuant     rebuild exactly and quantise;
//   kFormQuantEff  quantise the stage's bytes, which already hold W_eff.
constexpr int kFormAmax = 0, kFormAmaxKeep = 1, kFormQuant = 2, kFormQuantEff = 3;

// One 16-column block (columns 16b .. 16b + 15 of the lane's chunk) of both
// rows.  nu[h][t] = (u_t, u_t) of row h (see r4_pairs).  mx takes the
// NaN-propagating maximum of |e|; the quantising forms write the block's
// two packed words per row into out[h][2b], out[h][2b + 1] and return the
// four scale codes' contribution to the lane's scale word.  stage, g, c
// locate the lane's bytes for kFormAmaxKeep's write-back.
template <int kForm>
__device__ __forceinline__ uint32_t r4_block(const uint4 (&w)[2][4], const R4Row (&rw)[2],
                                             const uint64_t (&nu)[2][4],
                                             const float *__restrict__ vc, int b, float g_enc,
                                             const float *__restrict__ rcp_tab, bool ok,
                                             float &mx, uint32_t (&out)[2][4], uint8_t *stage,
                                             int g, int c) {
  constexpr bool kQuant = kForm == kFormQuant || kForm == kFormQuantEff;
  uint32_t bw[2][8];
  if constexpr (kForm == kFormQuantEff) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int pi = 0; pi < 8; ++pi) bw[h][pi] = word_of(w[h][2 * b + (pi >> 2)], pi & 3);
  } else {
    // Half a block (8 columns, 4 pairs) of both rows at a time, rank-outer:
    // eight independent fma chains per rank step.
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      uint64_t m[2][4] = {{0ull, 0ull, 0ull, 0ull}, {0ull, 0ull, 0ull, 0ull}};  // (+0, +0)
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float *vr = vc + t * 4 * kVtPitch + 16 * b + 8 * hb;
        const ulonglong2 va = *reinterpret_cast<const ulonglong2 *>(vr);
        const ulonglong2 vb = *reinterpret_cast<const ulonglong2 *>(vr + 4);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          m[h][0] = fma2(nu[h][t], va.x, m[h][0]);
          m[h][1] = fma2(nu[h][t], va.y, m[h][1]);
          m[h][2] = fma2(nu[h][t], vb.x, m[h][2]);
          m[h][3] = fma2(nu[h][t], vb.y, m[h][3]);
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int pi = 4 * hb + p;  // column pair within the block
          const uint32_t wd = word_of(w[h][2 * b + hb], p);
          if (kForm == kFormAmax) {
            const uint64_t e = fma2(pack2(-rw[h].s, -rw[h].s), bf16x2_to_f32x2(wd), m[h][p]);
            float elo, ehi;
            unpack2(e, elo, ehi);
            asm("max.NaN.abs.f32 %0, %0, %1, %2;" : "+f"(mx) : "f"(elo), "f"(ehi));
          } else {
            float mlo, mhi;
            unpack2(m[h][p], mlo, mhi);
            const float elo = __fmaf_rn(rw[h].s, bf16_lo(wd), -mlo);
            const float ehi = __fmaf_rn(rw[h].s, bf16_hi(wd), -mhi);
            bw[h][pi] = f32x2_to_bf16x2(ehi, elo);
            if (kForm == kFormAmaxKeep)
              asm("max.NaN.abs.f32 %0, %0, %1, %2;" : "+f"(mx) : "f"(elo), "f"(ehi));
          }
        }
      }
      if constexpr (kForm == kFormAmaxKeep) {
        uint8_t *box = stage + (c >> 1) * kR4BoxBytes;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          *reinterpret_cast<uint4 *>(box + (8 * h + g) * 128 +
                                     (((4 * (c & 1) + 2 * b + hb) ^ g) << 4)) =
              make_uint4(bw[h][4 * hb], bw[h][4 * hb + 1], bw[h][4 * hb + 2], bw[h][4 * hb + 3]);
      }
    }
  }
  uint32_t sword = 0;
  if (kQuant) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t sf = 0;
      out[h][2 * b] = out[h][2 * b + 1] = 0;
      if (ok) sf = quantize_block16(bw[h], g_enc, rcp_tab, out[h][2 * b], out[h][2 * b + 1]);
      sword |= sf << (16 * h + 8 * b);
    }
  }
  return sword;
}

// nu[h][t] = (u_t, u_t) of row h: the chain runs on u against the negated
// V tile, i.e. on -u against V.
__device__ __forceinline__ void r4_pairs(const R4Row (&rw)[2], uint64_t (&nu)[2][4]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float u[4] = {bf16_lo(rw[h].u01), bf16_hi(rw[h].u01), bf16_lo(rw[h].u23),
                        bf16_hi(rw[h].u23)};
#pragma unroll
    for (int t = 0; t < 4; ++t) nu[h][t] = pack2(u[t], u[t]);
  }
}

// The per-warp ring of one pass: which stage holds sequence position i, and
// the parity each stage's barrier completes with next (bit st).  With two
// stages, position i of a pass sits in stage (base + i) & 1; a pass that
// walks the previous pass's tiles backwards starts with base = iters - 1 on
// the two tiles that pass left resident.
struct R4Ring {
  uint8_t *ring, *rows;
  uint64_t *bars;
  uint32_t parity;
};
static_assert(kR4Stages == 2, "the resident-tile hand-over assumes two stages");

template <bool kPlain, typename TileOf>
__device__ __forceinline__ void r4_prime(const R4Maps &tm, R4Ring &rg, int64_t iters,
                                         TileOf tile_of, int64_t col0, int k, int lane) {
  if (lane == 0)
    for (int d = 0; d < kR4Stages && d < iters; ++d)
      r4_issue<kPlain>(tm, rg.ring + d * kR4StageBytes, rg.rows + d * kR4RowStride, &rg.bars[d],
               tile_of(d), col0, k);
  __syncwarp();
}

// One pass of a warp over its iters row tiles in the order tile_of(i).
// `resident` tiles at the start of the sequence are already in the ring
// (the previous pass waited for them, and left W_eff there, so the
// quantisation pass quantises them without a rebuild).  In the amax pass the
// tiles from position `keep_from` on stay resident for the quantisation
// pass, which gets their W_eff in the ring.  Returns false if a ring wait
// gave up (kDevTimeout is raised and the warp's other copies in flight are
// waited for, bounded).
template <bool kQuant, bool kKeep, bool kPlain, typename TileOf>
__device__ __forceinline__ bool r4_pass(const R4Maps &tm, R4Ring &rg, int64_t iters,
                                        int64_t base, int resident, int64_t keep_from,
                                        TileOf tile_of,
                                        int64_t col0, int k, int n, int64_t tiles_k,
                                        int64_t tk, const float *vc, int lane, float g_enc,
                                        const float *rcp_tab, bool ok, float &mx,
                                        uint32_t &mbits, uint8_t *__restrict__ packed,
                                        uint8_t *__restrict__ scales, volatile int *never,
                                        unsigned *status) {
  const int g = lane >> 2, c = lane & 3;
  const int64_t col = col0 + 32 * c;
  const bool live = col < k;
  for (int64_t i = 0; i < iters; ++i) {
    const int64_t tn = tile_of(i);
    const int st = int((base + i) & 1);
    if (i >= resident) {
      const bool arrived = core::mbar_wait(&rg.bars[st], (rg.parity >> st) & 1u, never);
      if (!__all_sync(0xFFFFFFFFu, arrived)) {
        if (lane == 0) {
          raise_status(status, kDevTimeout);
          const int other = st ^ 1;
          if (i + 1 < iters && i + 1 >= resident)
            core::mbar_wait(&rg.bars[other], (rg.parity >> other) & 1u, never);
        }
        return false;
      }
      rg.parity ^= 1u << st;
    }
    uint4 w[2][4];
    r4_read(rg.ring + st * kR4StageBytes, g, c, w);
    const R4Row rw[2] = {r4_row(rg.rows + st * kR4RowStride, g),
                         r4_row(rg.rows + st * kR4RowStride, 8 + g)};
    __syncwarp();
    if (lane == 0 && i + kR4Stages < iters)
      r4_issue<kPlain>(tm, rg.ring + st * kR4StageBytes, rg.rows + st * kR4RowStride,
                       &rg.bars[st],
               tile_of(i + kR4Stages), col0, k);
    uint32_t sword = 0;
    if (live) {
      uint8_t *stage = rg.ring + st * kR4StageBytes;
      uint32_t out[2][4];
      if (kPlain && !kQuant) {
        // largest magnitude as bf16 bit patterns with the sign cleared (a
        // NaN or an infinity sorts above every finite value), two per word
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            mbits = __vmaxu2(mbits, w[h][q].x & 0x7FFF7FFFu);
            mbits = __vmaxu2(mbits, w[h][q].y & 0x7FFF7FFFu);
            mbits = __vmaxu2(mbits, w[h][q].z & 0x7FFF7FFFu);
            mbits = __vmaxu2(mbits, w[h][q].w & 0x7FFF7FFFu);
          }
      } else if ((kPlain || kKeep) && kQuant && (kPlain || i < resident)) {
        const uint64_t nu[2][4] = {};
        sword |= r4_block<kFormQuantEff>(w, rw, nu, vc, 0, g_enc, rcp_tab, ok, mx, out, stage,
                                         g, c);
        sword |= r4_block<kFormQuantEff>(w, rw, nu, vc, 1, g_enc, rcp_tab, ok, mx, out, stage,
                                         g, c);
      } else {
        uint64_t nu[2][4];
        r4_pairs(rw, nu);
        if (kQuant) {
          sword |= r4_block<kFormQuant>(w, rw, nu, vc, 0, g_enc, rcp_tab, ok, mx, out, stage,
                                        g, c);
          sword |= r4_block<kFormQuant>(w, rw, nu, vc, 1, g_enc, rcp_tab, ok, mx, out, stage,
                                        g, c);
        } else if (kKeep && i >= keep_from) {
          r4_block<kFormAmaxKeep>(w, rw, nu, vc, 0, g_enc, rcp_tab, ok, mx, out, stage, g, c);
          r4_block<kFormAmaxKeep>(w, rw, nu, vc, 1, g_enc, rcp_tab, ok, mx, out, stage, g, c);
        } else {
          r4_block<kFormAmax>(w, rw, nu, vc, 0, g_enc, rcp_tab, ok, mx, out, stage, g, c);
          r4_block<kFormAmax>(w, rw, nu, vc, 1, g_enc, rcp_tab, ok, mx, out, stage, g, c);
        }
      }
      if (kQuant) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t row = tn * kTileRows + 8 * h + g;
          if (row < n)
            *reinterpret_cast<uint4 *>(packed + row * (k / 2) + col / 2) =
                make_uint4(out[h][0], out[h][1], out[h][2], out[h][3]);
        }
      }
    }
    if (kQuant) reinterpret_cast<uint32_t *>(scales + (tn * tiles_k + tk) * 128)[lane] = sword;
  }
  return true;
}

// The rank-4 passes.  kR4Amax: max |e| over the tensor into amax_bits[0] as
// bf16 bits with the sign cleared.  kR4Quant: the quantisation pass.  kR4Both:
// both in one cooperative launch -- every CTA folds its maximum into
// amax_bits[0], arrives on amax_bits[1] and waits (bounded) until all CTAs
// have; the quantisation pass then walks each warp's tiles backwards,
// starting on the two the amax pass left in its ring.  amax_bits[0..2] are
// zero at the start of the call, and the quantisation pass leaves them so
// (depart_and_clear).
// kR4BothKeep is kR4Both with the W_eff hand-over: the amax pass leaves the
// W_eff of each warp's last two tiles in its ring and the quantisation pass
// quantises them without a rebuild (worth it when a warp has few tiles; its
// extra code costs the main loop registers).
constexpr int kR4Amax = 0, kR4Quant = 1, kR4Both = 2, kR4BothKeep = 3;

// kPlain: the same passes over a bf16 weight W (tm.w0) quantised as it is,
// for aq_quantize_nvfp4: the amax pass takes the largest bf16 magnitude
// straight from the ring, the quantisation pass quantises the ring's bytes.
template <int kMode, bool kPlain = false, int kWarps = kR4Warps>
__global__ void __launch_bounds__(R4Geo<kWarps>::kThreads, R4Geo<kWarps>::kCtasPerSm)
    recon_r4_kernel(const __grid_constant__ R4Maps tm, const uint16_t *__restrict__ V, int n,
                    int k, uint8_t *__restrict__ packed,
                    uint8_t *__restrict__ scales, float *__restrict__ global_scale,
                    uint32_t *amax_bits, unsigned *status) {
  constexpr bool kBoth = kMode == kR4Both || kMode == kR4BothKeep;
  constexpr bool kKeep = kMode == kR4BothKeep;
  extern __shared__ uint8_t r4_smem_raw[];
  __shared__ float rcp_tab[128];
  __shared__ int never;  // abort flag of the bounded waits; nothing sets it
  __shared__ int grid_ok;
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(r4_smem_raw) + 1023) & ~uintptr_t(1023));
  const int wi = threadIdx.x >> 5, lane = threadIdx.x & 31, c = lane & 3;
  R4Ring rg{smem + wi * kR4Stages * kR4StageBytes,
            smem + R4Geo<kWarps>::kRowsOffset + wi * kR4Stages * kR4RowStride,
            reinterpret_cast<uint64_t *>(smem + R4Geo<kWarps>::kBarsOffset) + wi * kR4Stages,
            0u};
  float *vt = reinterpret_cast<float *>(smem + R4Geo<kWarps>::kRingBytes) + wi * kVtFloats;
  const int64_t tiles_k = ceil_div(k, kTileCols), tiles_n = ceil_div(n, kTileRows);
  const int64_t nw = int64_t(gridDim.x) * kWarps, w = int64_t(blockIdx.x) * kWarps + wi;
  const int64_t tk = w % tiles_k, col0 = tk * kTileCols, tn0 = w / tiles_k;
  const int64_t rows_in_flight = nw / tiles_k + (tk < nw % tiles_k ? 1 : 0);
  const int64_t iters = tn0 < tiles_n ? ceil_div(tiles_n - tn0, rows_in_flight) : 0;
  auto fwd = [&](int64_t i) { return tn0 + i * rows_in_flight; };
  auto rev = [&](int64_t i) { return tn0 + (iters - 1 - i) * rows_in_flight; };
  if (threadIdx.x == 0) never = 0;
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < kR4Stages; ++st) core::mbar_init(&rg.bars[st], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Launched as a programmatic dependent: the next call may start now, and
  // this one reads its inputs and the workspace only once the previous
  // kernel on the stream has finished.
  pdl_launch_dependents();
  pdl_wait();
  if (kMode == kR4Quant)
    r4_prime<kPlain>(tm, rg, iters, rev, col0, k, lane);
  else
    r4_prime<kPlain>(tm, rg, iters, fwd, col0, k, lane);
  if (!kPlain) stage_vt(V, col0, k, lane, vt);
  __syncthreads();
  const float *vc = vt + c * kVtPitch;
  bool ring_ok = true;

  if (kMode != kR4Quant) {
    float mx = 0.0f;
    // with the quantisation pass in the same launch, the last two tiles stay
    // resident with their W_eff
    const int64_t keep_from =
        kBoth ? (iters > kR4Stages ? iters - kR4Stages : 0) : iters;
    uint32_t mbits = 0;
    ring_ok = r4_pass<false, kKeep, kPlain>(tm, rg, iters, 0, 0, keep_from, fwd, col0, k, n,
                                            tiles_k, tk, vc, lane, 1.0f, rcp_tab, true, mx,
                                            mbits, nullptr, nullptr, &never, status);
    // bf16 bits of the largest |e|: a NaN stays a NaN pattern and an
    // infinity the infinity pattern, both at or above 0x7F80
    const uint32_t m = __float_as_uint(mx);
    uint32_t mb = kPlain ? max(mbits & 0xFFFFu, mbits >> 16)
                  : m >= 0x7F800000u ? (m >> 16) | (m > 0x7F800000u ? 0x40u : 0u)
                                     : uint32_t(f32_to_bf16_rn(mx));
    mb = block_max_u32<R4Geo<kWarps>::kThreads>(mb);
    if (threadIdx.x == 0) atomicMax(amax_bits, mb);
  }
  if (kMode == kR4Amax) return;

  if (kBoth) {
    // grid barrier: release this CTA's maximum, count it in, wait for all
    if (threadIdx.x == 0) {
      int ok_all = 1;
      __threadfence();
      atomicAdd(amax_bits + 1, 1u);
      unsigned seen = 0;
      for (unsigned it = 0;; ++it) {
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(seen) : "l"(amax_bits + 1)
                     : "memory");
        if (seen >= gridDim.x) break;
        if (it >= core::kSpinLimit) {
          raise_status(status, kDevTimeout);
          ok_all = 0;
          break;
        }
        __nanosleep(64);
      }
      grid_ok = ok_all;
    }
    __syncthreads();
    if (!grid_ok) return;
  }

  float g_enc = 1.0f, g_dec = 1.0f;
  uint32_t ab;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(ab) : "l"(amax_bits) : "memory");
  const bool ok = global_scales(ab, g_enc, g_dec);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *global_scale = ok ? g_dec : __int_as_float(0x7FC00000);
    if (!ok) raise_status(status, kDevRange);
  }
  fill_rcp_table(g_enc, rcp_tab);
  __syncthreads();
  depart_and_clear(amax_bits);
  if (!ring_ok) return;
  float unused = 0.0f;
  const int resident = kBoth ? int(iters < kR4Stages ? iters : kR4Stages) : 0;
  const int64_t base = kBoth ? iters - 1 : 0;
  uint32_t unused_bits = 0;
  r4_pass<true, kKeep, kPlain>(tm, rg, iters, base, resident, iters, rev, col0, k, n, tiles_k,
                               tk, vc, lane, g_enc, rcp_tab, ok, unused, unused_bits, packed,
                               scales, &never, status);
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
  // Launched with programmatic dependent launch: the MMA kernel that
  // follows may start now (it waits for this grid before it reads the
  // quantised activations); x and the outputs wait for the previous kernel.
  pdl_launch_dependents();
  pdl_wait();
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
  __shared__ float rcp_tab[128];
  fill_rcp_table(g_enc, rcp_tab);
  __syncthreads();
  for (int b = threadIdx.x; b < k / kBlock; b += kThreads) {
    const uint4 v0 = __ldg(reinterpret_cast<const uint4 *>(xr + b * kBlock));
    const uint4 v1 = __ldg(reinterpret_cast<const uint4 *>(xr + b * kBlock) + 1);
    const uint32_t bw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t lo = 0, hi = 0, sf = 0;
    if (ok) sf = quantize_block16(bw, g_enc, rcp_tab, lo, hi);
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

// The per-element fused form (ranks other than 4, or U, s or V not 16-byte
// aligned): the amax pass, then the quantisation pass, both grid-stride.
template <int R>
static void quantize_pass(const uint16_t *W, const float *s, const uint16_t *U,
                          const uint16_t *V, int r, int n, int k,
                          const aq_nvfp4_weight &out, uint32_t *amax, const DeviceInfo &dev,
                          cudaStream_t st) {
  const int cap = dev.sms * 8;
  const int ga = grid_for(int64_t(n) * (k / 8), kThreads, cap);
  amax_fused_kernel<R><<<ga, kThreads, 0, st>>>(W, s, U, V, n, k, r, amax);
  const int64_t tiles = ceil_div(n, kTileRows) * ceil_div(k, kTileCols);
  const int g = grid_for(tiles, kThreads / 32, cap);
  quantize_kernel<R><<<g, kThreads, 0, st>>>(W, s, U, V, n, k, r, out.packed, out.scales,
                                             out.global_scale, amax, dev.status);
}

// Rank 4: 16 warps per SM (fewer for a small tensor), so that every SM
// carries the same number of warps; every tile column needs a warp, and
// when that takes more CTAs than fit on the GPU at once the two passes run
// as two launches, else as one cooperative launch (kR4Both).
template <int kMode, bool kPlain = false, int kWarps = kR4Warps>
static cudaError_t r4_smem_attr(int device) {
  static bool done[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (device >= 0 && device < 64 && done[device]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(recon_r4_kernel<kMode, kPlain, kWarps>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             R4Geo<kWarps>::kSmemBytes);
  if (e == cudaSuccess && device >= 0 && device < 64) done[device] = true;
  return e;
}

// CTAs of a cooperative form that can be resident at once (0 if unknown).
template <int kMode, bool kPlain = false, int kWarps = kR4Warps>
static int64_t r4_both_capacity(const DeviceInfo &dev) {
  static int per_sm[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (dev.ordinal < 0 || dev.ordinal >= 64) return 0;
  if (per_sm[dev.ordinal] == 0) {
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &nb, recon_r4_kernel<kMode, kPlain, kWarps>, R4Geo<kWarps>::kThreads,
            R4Geo<kWarps>::kSmemBytes) != cudaSuccess)
      nb = -1;
    per_sm[dev.ordinal] = nb > 0 ? nb : -1;
  }
  return per_sm[dev.ordinal] > 0 ? int64_t(per_sm[dev.ordinal]) * dev.sms : 0;
}

// The W_eff hand-over pays while a warp has at most this many row tiles.
constexpr int64_t kR4KeepMaxTiles = 8;

// CTAs of `warps` warps for a weight of tiles_n x tiles_k row tiles: one
// tile per warp up to 16 warps per SM, and at least one warp per tile column.
static int64_t r4_grid(int64_t tiles_n, int64_t tiles_k, int warps, const DeviceInfo &dev) {
  int64_t G = ceil_div(tiles_k * tiles_n, warps);
  if (G > int64_t(dev.sms) * (16 / warps)) G = int64_t(dev.sms) * (16 / warps);
  if (G < ceil_div(tiles_k, warps)) G = ceil_div(tiles_k, warps);
  return G;
}

// Both passes over a weight of [n, k]: kPlain for a bf16 W in tm.w0, else
// the rank-4 theta bundle (tm.w0 = W0, tm.u, tm.s, V).
template <bool kPlain>
static cudaError_t r4_launch(const R4Maps &tm, const uint16_t *V, int n, int k,
                             const aq_nvfp4_weight &out, uint32_t *amax, const DeviceInfo &dev,
                             cudaStream_t st) {
  cudaError_t e = r4_smem_attr<kR4Amax, kPlain>(dev.ordinal);
  if (e == cudaSuccess) e = r4_smem_attr<kR4Quant, kPlain>(dev.ordinal);
  if (e == cudaSuccess) e = r4_smem_attr<kR4Both, kPlain>(dev.ordinal);
  if (e == cudaSuccess && !kPlain) e = r4_smem_attr<kR4BothKeep>(dev.ordinal);
  if (e == cudaSuccess && !kPlain) e = r4_smem_attr<kR4Both, false, kR4WideWarps>(dev.ordinal);
  if (e != cudaSuccess) return e;
  const int64_t tiles_k = ceil_div(k, kTileCols), tiles_n = ceil_div(n, kTileRows);
  const int64_t G = r4_grid(tiles_n, tiles_k, kR4Warps, dev);
  const int g = int(G);
  uint8_t *packed = out.packed, *scales = out.scales;
  float *gs = out.global_scale;
  unsigned *status = dev.status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g);
  cfg.blockDim = dim3(R4Geo<kR4Warps>::kThreads);
  cfg.dynamicSmemBytes = R4Geo<kR4Warps>::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  // the most row tiles a warp gets: its tile column's tiles over the
  // column's (fewest) warps
  const int64_t most_tiles = ceil_div(tiles_n, G * kR4Warps / tiles_k);
  if (!kPlain && most_tiles <= kR4KeepMaxTiles && g <= r4_both_capacity<kR4BothKeep>(dev)) {
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, recon_r4_kernel<kR4BothKeep>, tm, V, n, k, packed, scales,
                              gs, amax, status);
  }
  if (!kPlain) {
    const int64_t gw = r4_grid(tiles_n, tiles_k, kR4WideWarps, dev);
    if (gw <= r4_both_capacity<kR4Both, false, kR4WideWarps>(dev)) {
      cudaLaunchConfig_t wide = cfg;
      wide.gridDim = dim3(unsigned(gw));
      wide.blockDim = dim3(R4Geo<kR4WideWarps>::kThreads);
      wide.dynamicSmemBytes = R4Geo<kR4WideWarps>::kSmemBytes;
      wide.numAttrs = 2;
      return cudaLaunchKernelEx(&wide, recon_r4_kernel<kR4Both, false, kR4WideWarps>, tm, V, n,
                                k, packed, scales, gs, amax, status);
    }
  }
  if (g <= r4_both_capacity<kR4Both, kPlain>(dev)) {
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, recon_r4_kernel<kR4Both, kPlain>, tm, V, n, k, packed,
                              scales, gs, amax, status);
  }
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, recon_r4_kernel<kR4Amax, kPlain>, tm, V, n, k,
                         static_cast<uint8_t *>(nullptr), static_cast<uint8_t *>(nullptr),
                         static_cast<float *>(nullptr), amax, status);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, recon_r4_kernel<kR4Quant, kPlain>, tm, V, n, k, packed,
                            scales, gs, amax, status);
}

static cudaError_t quantize_pass_r4(const uint16_t *W, const float *s, const uint16_t *U,
                                    const uint16_t *V, int n, int k,
                                    const aq_nvfp4_weight &out, uint32_t *amax,
                                    const DeviceInfo &dev, cudaStream_t st) {
  R4Maps tm;
  if (!core::encode_bf16_rows_map(W, n, k, kTileRows, &tm.w0) ||
      !core::encode_bytes_1d(U, uint64_t(n) * 8, kTileRows * 8, &tm.u) ||
      !core::encode_bytes_1d(s, uint64_t(n) * 4, kTileRows * 4, &tm.s))
    return cudaErrorInvalidValue;
  return r4_launch<false>(tm, V, n, k, out, amax, dev, st);
}

// A bf16 weight quantised as it is, through the same passes.
static cudaError_t quantize_pass_plain(const uint16_t *W, int n, int k,
                                       const aq_nvfp4_weight &out, uint32_t *amax,
                                       const DeviceInfo &dev, cudaStream_t st) {
  R4Maps tm;
  memset(&tm, 0, sizeof(tm));
  if (!core::encode_bf16_rows_map(W, n, k, kTileRows, &tm.w0)) return cudaErrorInvalidValue;
  return r4_launch<true>(tm, nullptr, n, k, out, amax, dev, st);
}

cudaError_t launch_quantize(const uint16_t *W, const float *s, const uint16_t *U,
                            const uint16_t *V, int r, bool fused, int n, int k,
                            const aq_nvfp4_weight &out, void *ws, const DeviceInfo &dev,
                            cudaStream_t st) {
  // [0] amax bits, [1] grid arrivals, [2] departures: zero on entry, and
  // zero again when the quantisation pass is done
  uint32_t *amax = static_cast<uint32_t *>(ws);
  if (!fused)
    return quantize_pass_plain(W, n, k, out, amax, dev, st);
  else if (r == 4 && ((reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(U) |
                        reinterpret_cast<uintptr_t>(s)) & 15u) == 0)
    return quantize_pass_r4(W, s, U, V, n, k, out, amax, dev, st);
  else if (r == 0)
    quantize_pass<0>(W, s, U, V, r, n, k, out, amax, dev, st);
  else if (r == 4 && (reinterpret_cast<uintptr_t>(V) & 7u) == 0)
    quantize_pass<4>(W, s, U, V, r, n, k, out, amax, dev, st);
  else
    quantize_pass<-1>(W, s, U, V, r, n, k, out, amax, dev, st);
  return cudaGetLastError();
}

cudaError_t launch_act_quant(const uint16_t *x, int m, int k, uint8_t *packed, uint8_t *scales,
                             int scale_pitch, float *g_dec, const DeviceInfo &dev,
                             cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(m);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, act_quant_kernel, x, k, packed, scales, scale_pitch, g_dec,
                            dev.status);
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
