// lowrank.cu -- the runtime low-rank GEMV: y = s * (W0_hat x) + U (V^T x)
// for a quantised block W0 shared across a band of layers, a per-row scale
// s and a rank-r correction U V^T, evaluated without rebuilding the weight.
//
// AttnQuant docs, "Throughput", "The runtime reconstruction path does not
// reach dense parity" (the path that rebuilds W0 and the low-rank delta in
// the graph on every forward pass), and "GPU acceleration", "How the pieces
// fit" (the custom op that fuses the shared-block dot product with the
// low-rank delta, no intermediate materialised); landing page, "How it
// works" for the theta bundle (W0, s, U, V).
//
// Two launches on the stream: vx_kernel writes t = V^T x (fp32 [m, r]) into
// the workspace, then the register-decode GEMV streams W0_hat and applies
// s and U t in its epilogue (out_value in gemv_core.cuh).  The GEMV is
// launched with programmatic dependent launch behind vx_kernel: its weight
// stream starts at once and its consumers read t after the wait.
#include "gemv_core.cuh"

namespace aq {

using namespace core;

namespace {

constexpr int kVxThreads = 512;
constexpr int kMaxRank = 16;
constexpr int kMaxChunks = 32;

// Chunks of k per token: enough CTAs that each thread sums one or two k.
__host__ __device__ __forceinline__ int vx_chunks(int k) {
  const int c = (k + kVxThreads - 1) / kVxThreads;
  return c < 1 ? 1 : (c > kMaxChunks ? kMaxChunks : c);
}

// Grid (chunks, m): CTA (c, tok) sums V[k, q] x[tok, k] over its fixed
// k-range in fp32 (threads by a fixed stride, warps by a fixed butterfly,
// the CTA over warps in order) and stores the chunk partial; the CTA that
// takes the token's last ticket adds the partials in chunk order into
// t[tok, q] and clears the ticket.  The result does not depend on timing.
__global__ void __launch_bounds__(kVxThreads)
    vx_kernel(const uint16_t *__restrict__ V, const uint16_t *__restrict__ x, int k, int r,
              float *__restrict__ t, float *__restrict__ t_part, uint32_t *__restrict__ tickets) {
  pdl_launch_dependents();  // the GEMV may start streaming its weights now
  pdl_wait();               // x may come from the previous kernel
  __shared__ float part[kVxThreads / 32][kMaxRank];
  __shared__ int last;
  const int chunks = gridDim.x, c = blockIdx.x, tok = blockIdx.y;
  const int per = (k + chunks - 1) / chunks;
  const int j0 = c * per, j1 = min(k, j0 + per);
  const uint16_t *xr = x + int64_t(tok) * k;
  float acc[kMaxRank];
#pragma unroll
  for (int q = 0; q < kMaxRank; ++q) acc[q] = 0.0f;
  for (int j = j0 + threadIdx.x; j < j1; j += kVxThreads) {
    const float xv = __uint_as_float(uint32_t(xr[j]) << 16);
    const uint16_t *vr = V + int64_t(j) * r;
#pragma unroll
    for (int q = 0; q < kMaxRank; ++q)
      if (q < r) acc[q] = __fmaf_rn(__uint_as_float(uint32_t(vr[q]) << 16), xv, acc[q]);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < kMaxRank; ++q) {
    if (q >= r) break;
    float v = acc[q];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    if (lane == 0) part[warp][q] = v;
  }
  __syncthreads();
  if (threadIdx.x < r) {
    float sum = 0.0f;
    for (int w = 0; w < kVxThreads / 32; ++w) sum = __fadd_rn(sum, part[w][threadIdx.x]);
    t_part[(int64_t(tok) * chunks + c) * r + threadIdx.x] = sum;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(tickets + tok) : "memory");
    last = old == unsigned(chunks - 1);
  }
  __syncthreads();
  if (last) {
    if (threadIdx.x < r) {
      float sum = 0.0f;
      for (int cc = 0; cc < chunks; ++cc)
        sum = __fadd_rn(sum, __ldcg(t_part + (int64_t(tok) * chunks + cc) * r + threadIdx.x));
      t[tok * r + threadIdx.x] = sum;
    }
    if (threadIdx.x == 0) tickets[tok] = 0;
  }
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// Workspace of the low-rank GEMV: the GEMV's, then t [m, r], the chunk
// partials [m, chunks, r] and one ticket per token (zero between calls).
struct LrLayout {
  size_t t_off, part_off, ticket_off, bytes;
};
LrLayout lr_layout(int n, int k, int m, int r, const DeviceInfo &dev) {
  const int rr = r > 0 ? r : 1;
  LrLayout l;
  l.t_off = align256(gemv_workspace_bytes(n, k, dev));
  l.part_off = l.t_off + align256(size_t(m) * rr * 4);
  l.ticket_off = l.part_off + align256(size_t(m) * vx_chunks(k) * rr * 4);
  l.bytes = l.ticket_off + align256(size_t(m) * 4);
  return l;
}

}  // namespace

size_t gemv_lowrank_workspace_bytes(int n, int k, int m, int r, const DeviceInfo &dev) {
  return lr_layout(n, k, m, r, dev).bytes;
}

cudaError_t launch_gemv_lowrank(const aq_nvfp4_weight &w0, const float *s, const uint16_t *U,
                                const uint16_t *V, int r, const uint16_t *x, int m,
                                uint16_t *y, void *ws, bool pdl, const DeviceInfo &dev,
                                cudaStream_t st) {
  const LrLayout l = lr_layout(w0.n, w0.k, m, r, dev);
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  float *t = reinterpret_cast<float *>(wsb + l.t_off);
  if (r > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(vx_chunks(w0.k), m);
    cfg.blockDim = dim3(kVxThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, vx_kernel, V, x, w0.k, r, t,
                                       reinterpret_cast<float *>(wsb + l.part_off),
                                       reinterpret_cast<uint32_t *>(wsb + l.ticket_off));
    if (e != cudaSuccess) return e;
  }
  const LowRank lr{s, U, t, r};
  // behind vx_kernel (or, for r = 0, behind the caller's previous work when
  // pdl is asked for)
  return launch_gemv_regdecode(w0, x, m, y, ws, r > 0 || pdl, dev, st, nullptr, &lr);
}

}  // namespace aq
