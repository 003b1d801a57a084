// 5th-generation tensor-core primitives (tcgen05: MMAs with shared-memory
// operands and accumulators in tensor memory), written from the PTX ISA.
//
// Shared-memory operand tiles use the 128-byte swizzle: rows of 128 bytes
// (64 bf16), grouped in 8-row atoms of 1024 bytes that start 1024-byte
// aligned; the 16-byte chunk c of row r of an atom is stored at chunk
// c ^ (r & 7). A "K-major" tile holds rows of the non-reduced dimension (M or
// N) with 64 reduction-dimension elements each; an "MN-major" tile holds rows
// of the reduction dimension with 64 M (or N) elements each, and a 128-wide
// operand is two such 64-wide tiles `atom_bytes` apart.
//
// Accumulators for M = 128 live in TMEM with row i in lane i and column j in
// column (base + j); warp w of a warpgroup reads lanes [32 (w % 4), +32).
#pragma once

#include <stdint.h>

#include "gdn_mma.cuh"

namespace gdn {

// Byte offset of element (r, c) (c < 128) of a swizzled tile whose 64-wide
// halves are `half_bytes` apart.
__device__ __forceinline__ uint32_t sw128(int r, int c, uint32_t half_bytes) {
  return (uint32_t)(c >> 6) * half_bytes + (uint32_t)r * 128u +
         ((((uint32_t)(c & 63) >> 3) ^ ((uint32_t)r & 7u)) << 4) + (uint32_t)(c & 7) * 2u;
}

// Shared-memory matrix descriptor: start address, leading-dimension byte
// offset (MN-major: distance between 64-wide tiles; unused for K-major),
// stride-dimension byte offset (distance between 8-row atoms), descriptor
// version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 accumulator,
// A / B major-ness (0 = K-major, 1 = MN-major), N and M.
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A * B, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate));
}

// Arrives once on `bar` when every MMA this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {  // one warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_u32(slot)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // one warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (load and wait in
// one statement, so no use of the registers can be scheduled before the wait).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace gdn

namespace gdn {
// 1-D bulk copy shared -> global (16-byte aligned, size a multiple of 16),
// tracked by this thread's bulk-group; the smem source must be made visible
// to the async proxy first (fence_proxy_async_smem + barrier).
__device__ __forceinline__ void bulk_s2g(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(gdst),
               "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// Waits until the committed bulk stores of this thread have read their smem sources.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
}  // namespace gdn

namespace gdn {
// 4-D tiled tensor copy global -> shared (TMA), completing its bytes on `bar`.
// `tmap` is the address of a __grid_constant__ CUtensorMap kernel parameter;
// c0 is the innermost coordinate (its byte offset must be a multiple of 16).
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int c0, int c1, int c2,
                                            int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar))
      : "memory");
}
}  // namespace gdn

namespace gdn {
// 3-D tiled tensor copy global -> shared, completing its bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace gdn
