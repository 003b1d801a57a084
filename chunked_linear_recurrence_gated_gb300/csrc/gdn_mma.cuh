// Warp-level bf16 tensor-core primitives (mma.sync m16n8k16, ldmatrix,
// cp.async) used by the register-resident kernels of the bf16 path.
//
// Fragment layouts of mma.m16n8k16 (g = lane / 4, t = lane % 4):
//   A (16 x 16, row):  a0 (g, 2t..2t+1)   a1 (g+8, 2t..)   a2 (g, 2t+8..)   a3 (g+8, 2t+8..)
//   B (16 x 8, col):   b0 (k 2t..2t+1, n g)                 b1 (k 2t+8.., n g)
//   C (16 x 8, f32):   c0,c1 (g, 2t..2t+1)                  c2,c3 (g+8, 2t..2t+1)
// A C fragment pair covering columns [16j, 16j+16) is therefore an A fragment
// of a k16 slice once packed to bf16, which lets a product's output feed the
// next product without leaving registers.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace gdn {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Transposing store of four 8x8 bf16 matrices held as MMA accumulator pairs:
// lanes 8m..8m+7 give the row addresses (16-byte aligned) of stored matrix m,
// whose row i is column i of fragment r[m].
__device__ __forceinline__ void stsm_x4_t(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                          uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(addr),
               "r"(r0), "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}

__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}

// A fragment (16 x 16) from a row-major bf16 tile: rows [r0, r0+16), cols [c0, c0+16).
__device__ __forceinline__ void lda_rm(uint32_t* a, const __nv_bfloat16* base, int ld, int r0,
                                       int c0) {
  const int l = threadIdx.x & 31;
  const __nv_bfloat16* p = base + (r0 + (l & 7) + ((l >> 3) & 1) * 8) * ld + c0 + (l >> 4) * 8;
  ldsm_x4(smem_u32(p), a[0], a[1], a[2], a[3]);
}

// A fragment (16 x 16) of M^T where M is stored row-major: A[m][k] = M[k][m],
// A rows m in [m0, m0+16), cols k in [k0, k0+16).
__device__ __forceinline__ void lda_tr(uint32_t* a, const __nv_bfloat16* base, int ld, int m0,
                                       int k0) {
  const int l = threadIdx.x & 31;
  // matrices: (k0, m0) (k0, m0+8) (k0+8, m0) (k0+8, m0+8) in stored coordinates
  const int mat = l >> 3;
  const int krow = k0 + (l & 7) + (mat >> 1) * 8;
  const int mcol = m0 + (mat & 1) * 8;
  ldsm_x4_t(smem_u32(base + krow * ld + mcol), a[0], a[1], a[2], a[3]);
}

// B fragments for one k16 step of two n8 tiles from storage [n][k]:
// rows n in [n0, n0+16), k in [k0, k0+16). b[0..1] = tile n0, b[2..3] = tile n0+8.
__device__ __forceinline__ void ldb_nk_x2n(uint32_t* b, const __nv_bfloat16* base, int ld, int n0,
                                           int k0) {
  const int l = threadIdx.x & 31;
  const int mat = l >> 3;
  const __nv_bfloat16* p = base + (n0 + (l & 7) + (mat >> 1) * 8) * ld + k0 + (mat & 1) * 8;
  ldsm_x4(smem_u32(p), b[0], b[1], b[2], b[3]);
}

// B fragments for one k16 step of two n8 tiles from storage [k][n] (row-major,
// n contiguous): k in [k0, k0+16), n in [n0, n0+16). b[0..1] = tile n0, b[2..3] = n0+8.
__device__ __forceinline__ void ldb_kn_x2n(uint32_t* b, const __nv_bfloat16* base, int ld, int k0,
                                           int n0) {
  const int l = threadIdx.x & 31;
  const int mat = l >> 3;
  const __nv_bfloat16* p = base + (k0 + (l & 7) + (mat & 1) * 8) * ld + n0 + (mat >> 1) * 8;
  ldsm_x4_t(smem_u32(p), b[0], b[1], b[2], b[3]);
}

// cp.async of 16 bytes, zero-filling when `valid` is false.
__device__ __forceinline__ void cp16(void* smem, const void* gmem, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)),
               "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

}  // namespace gdn

namespace gdn {

// ---------------------------------------------------------------- mbarrier + bulk copies
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
// Makes mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the barrier phase with the given parity. Gives up after `limit` SM
// clock cycles (default about two seconds), sets *abort and returns false (the
// caller then skips its work but keeps executing every barrier, so the kernel
// still terminates).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          long long limit = (1ll << 32)) {
  const int aborted = *abort;  // read alongside the first try, not before it
  const bool done = mbar_try_wait(bar, parity);
  if (aborted) return false;
  if (done) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      *abort = 1;
      return false;
    }
  }
  return true;
}
// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16),
// completing `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Named barrier over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace gdn

namespace gdn {
// Arrives on `bar` once all of this thread's prior cp.async copies have landed
// (the barrier's expected count must include this arrival).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar))
               : "memory");
}
}  // namespace gdn

namespace gdn {
// ---------------------------------------------------------------- TF32 warp-level MMA
// mma.m16n8k8 with tf32 inputs (fp32 storage, 10-bit mantissa) and fp32
// accumulation. Fragments (g = lane / 4, t = lane % 4):
//   A (16 x 8): a0 (g, t) a1 (g+8, t) a2 (g, t+4) a3 (g+8, t+4)
//   B (8 x 8):  b0 (k t, n g) b1 (k t+4, n g)
//   C (16 x 8): c0, c1 (g, 2t..2t+1) c2, c3 (g+8, 2t..2t+1)
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
}  // namespace gdn
