// tc_ptx.cuh -- inline-PTX wrappers for the 5th-generation tensor cores
// (tcgen05) on sm_103a: tensor-memory allocation, loads and stores, the
// block-scaled fp4 MMA and its shared-memory operand descriptors.
//
// Facts these wrappers rely on, checked on GB300 with an in-bounds probe of
// known operands against an fp64 host product:
//  * kind::mxf4nvf4 with scale_vec::4X takes E2M1 operands packed two per
//    byte (lower k in the low nibble) and one E4M3 scale per 16 k.
//  * A K-major operand tile with 128-byte rows and the 128-byte swizzle (the
//    layout a TMA box of 128 B x rows with CU_TENSOR_MAP_SWIZZLE_128B writes)
//    is described by start address, stride 1024 B between 8-row groups; the
//    k-th 64-element step starts 32 B further.
//  * The scales of one MMA (4 per row: k blocks 0..3 of its 64 columns) sit
//    in a group of 4 TMEM columns at a 4-aligned column c0.  Row r's four
//    scale bytes are the 32-bit cell at column c0 + r / 32, in every lane
//    whose index is r mod 32 (all four 32-lane quarters hold the copy).  The
//    same holds for the B operand with its column index n in place of r.
//  * The accumulator of an M = 128 MMA holds row r in TMEM lane r and output
//    column n in column d0 + n (fp32).
//  * tcgen05.cp 32x128b.warpx4 copies a 512-byte shared-memory atom (32 rows
//    of 16 B, no swizzle, 8-row core matrices 128 B apart) into 4 columns of
//    every 32-lane quarter: lane 32q + i, column c0 + c receives atom bytes
//    16i + 4c .. 16i + 4c + 3.  So an MMA's 128 x 4 scales, row r's four
//    bytes at atom offset (r % 32) * 16 + (r / 32) * 4, land exactly in the
//    layout above.
#pragma once

#include <cstdint>

namespace aq {
namespace tcx {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory descriptor of a K-major operand tile with 128-byte rows,
// 128-byte swizzle, 8-row groups 1024 B apart.  `addr` must lie in a
// 1024-byte aligned tile, offset by a multiple of 32 B within a row.
__device__ __forceinline__ uint64_t desc_k_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= uint64_t((addr & 0x3FFFFu) >> 4);  // start address
  d |= uint64_t(1) << 16;                 // leading offset (unused with this swizzle)
  d |= uint64_t(1024 >> 4) << 32;         // stride between 8-row groups
  d |= uint64_t(1) << 46;                 // descriptor version
  d |= uint64_t(2) << 61;                 // 128-byte swizzle
  return d;
}

// Instruction descriptor: block-scaled E2M1 x E2M1, E4M3 scales, fp32
// accumulator, both operands K-major, M = 128, N = n (a multiple of 16).
__host__ __device__ __forceinline__ uint32_t idesc_nvf4(int n) {
  return (1u << 7) | (1u << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(128 >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes become visible to the tensor core.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory descriptor of a copy atom: no swizzle, 8-row core matrices
// of 16-byte rows, 128 B apart (leading and stride offsets both 128 B).
__device__ __forceinline__ uint64_t desc_atom(uint32_t addr) {
  return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t(128 >> 4) << 16) |
         (uint64_t(128 >> 4) << 32) | (uint64_t(1) << 46);
}

// Shared-memory atom -> 4 tensor-memory columns (replicated over the four
// lane quarters); issued by one thread, ordered with its MMAs.
__device__ __forceinline__ void cp_atom(uint32_t taddr, uint64_t src_desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(src_desc)
               : "memory");
}

// D (+)= A * B with block scales; issued by one thread.
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
      "[%0], %1, %2, %3, [%5], [%6], p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u), "r"(sfa_tmem),
      "r"(sfb_tmem)
      : "memory");
}

// The mbarrier completes one arrival once every MMA this thread issued
// before has finished.
__device__ __forceinline__ void commit_to(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// 16 consecutive 32-bit columns of this warp's 32 lanes (lane = thread).
__device__ __forceinline__ void st_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void ld_x16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace tcx
}  // namespace aq
