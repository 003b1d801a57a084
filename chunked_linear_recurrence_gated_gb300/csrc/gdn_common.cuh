// Shared device-side definitions of the GDN chunk kernels: sequence/block
// maps, workspace views and element loads. Internal to the library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

// Kernel-level block length: the blocks b_{i,j} inside a chunk (StateFlow
// review, "Assumptions & free parameters"). Blocks are anchored at the start
// of every sequence of a call, so a split at a multiple of BT leaves every
// block, and therefore every result, unchanged.
constexpr int BT = 64;

// Where the blocks of a call live. Fixed-length calls have B sequences of T
// tokens each (token n of sequence b is row b*T + n); varlen calls read the
// sequence offsets from cu_seqlens and the block tables the prep kernel wrote.
struct SeqMap {
  const int* cu;       // varlen: device cu_seqlens [nseq + 1]; fixed: nullptr
  const int* blk0;     // varlen: first global block of each sequence [nseq + 1]
  const int* blk_seq;  // varlen: owning sequence of each global block (-1 = none)
  const int* order;    // varlen: sequences longest first (the chains' CTA order); fixed: nullptr
  int nseq;
  int T_fixed;         // fixed: tokens per sequence
  int nblk_fixed;      // fixed: blocks per sequence
  int nblk_cap;        // global blocks launched by the per-block kernels
  int H;
  long long T_total;   // tokens of the call (B * T, or the packed total)
};

struct BlockInfo {
  int seq, tok0, len, lb;
};

__device__ __forceinline__ bool block_info(const SeqMap& m, int gb, BlockInfo& bi) {
  if (m.cu == nullptr) {
    const int s = gb / m.nblk_fixed;
    const int lb = gb - s * m.nblk_fixed;
    bi.seq = s;
    bi.lb = lb;
    bi.tok0 = s * m.T_fixed + lb * BT;
    bi.len = min(BT, m.T_fixed - lb * BT);
    return bi.len > 0;
  }
  const int s = m.blk_seq[gb];
  if (s < 0) return false;
  const int lb = gb - m.blk0[s];
  const int t0 = m.cu[s] + lb * BT;
  bi.seq = s;
  bi.lb = lb;
  bi.tok0 = t0;
  bi.len = min(BT, m.cu[s + 1] - t0);
  return bi.len > 0;
}

struct SeqInfo {
  int tok0, len, blk0, nblk;
};

__device__ __forceinline__ SeqInfo seq_info(const SeqMap& m, int s) {
  if (m.cu == nullptr) return {s * m.T_fixed, m.T_fixed, s * m.nblk_fixed, m.nblk_fixed};
  const int t0 = m.cu[s], t1 = m.cu[s + 1];
  const int b0 = m.blk0[s], b1 = m.blk0[s + 1];
  if (t1 < t0 || b1 < b0) return {t0, 0, b0, 0};
  return {t0, t1 - t0, b0, b1 - b0};
}

// Device-side status codes written into the workspace status word.
enum : int { DEV_OK = 0, DEV_BAD_CU_SEQLENS = 1, DEV_TIMEOUT = 2 };

// Workspace views (fp32 intermediates of the SIMT kernels). Indexed by
// bh = global_block * H + head.
struct SimtWs {
  int* status;
  float* gam;  // [nblk, H, BT]     block-local cumulative log-decay
  float* W;    // [nblk, H, BT, dk] W = T diag(beta Gamma) K
  float* U;    // [nblk, H, BT, dv] U = T diag(beta) V
  float* Hb;   // [nblk, H, dk, dv] state at the start of the block
  float* Vn;   // [nblk, H, BT, dv] V^new = U - W Hb
  float* Tm;   // [nblk, H, BT, BT] T = (I + A)^-1            (backward)
  float* dH;   // [nblk, H, dk, dv] state gradient after the block (backward)
  float* dVn;  // [nblk, H, BT, dv] gradient of V^new      (backward)
};

// Workspace views of the bf16 tensor-core kernels (bh = global_block * H + head).
// Pre writes W, U and QKM with padded rows so that each lands in the chain's
// padded shared-memory tiles with a single bulk copy.
constexpr int TC_LDK = 136;   // padded row of 128-wide bf16 tiles
constexpr int TC_LD64 = 72;   // padded row of 64-wide bf16 tiles
constexpr int TC_LDU = 16;    // row of a 16-column U tile (two 16-byte chunks)
// Element (t, c) of a 16-column tile: the two 16-byte chunks of row t swap
// places when bit 2 of t is set, so 8 consecutive rows read at one chunk hit
// 8 different bank groups without padding.
__host__ __device__ constexpr int u_tile_off(int t, int c) {
  return t * TC_LDU + (((c >> 3) ^ ((t >> 2) & 1)) << 3) + (c & 7);
}
constexpr int TC_DEC_ROWS = 4;  // per-block vectors in TcWs::dec
struct TcWs {
  int* status;
  float* dec;            // [nblk, H, 4, BT]   Gamma_r, e^{gamma_C - gamma_r}, gamma_r, beta_r
                         //                    (beta_r = 0 past the end of the block)
  __nv_bfloat16* W;      // [nblk, H, BT, TC_LDK]          W = T diag(beta Gamma) K: the first 2 x BT x 64
                         //                    elements of each block-head hold two 128-byte-swizzled
                         //                    [t][64 key] tiles (sw128 of gdn_umma.cuh)
  __nv_bfloat16* U;      // [nblk, H, dv/16, BT, TC_LDU]   U = T diag(beta) V, tile-major (u_tile_off)
  __nv_bfloat16* QKM;    // [nblk, H, BT, TC_LD64]         Q K^T * Mask (j <= r): the first BT x 64
                         //                    elements of each block-head hold one 128-byte-swizzled
                         //                    [t][j] tile (sw128 of gdn_umma.cuh)
  __nv_bfloat16* Kp;     // [nblk, H, BT, TC_LDK]          K~ = e^{gamma_C - gamma} K, as W (zero past the end)
  __nv_bfloat16* Qp;     // [nblk, H, BT, TC_LDK]          Q~ = e^{gamma} Q: the first 2 x BT x 64 elements
                         //                    of each block-head hold two 128-byte-swizzled [t][64 key]
                         //                    tiles (keys 0-63, 64-127; zero past the end)
  __nv_bfloat16* T;      // [nblk, H, BT, BT]      (I + A)^-1          (backward)
  __nv_bfloat16* KKM;    // [nblk, H, BT, TC_LD64] K K^T * Mask, strictly lower, as QKM (backward)
  __nv_bfloat16* HbT;    // [nblk, H, dv, 128]     H_b^T               (backward)
  __nv_bfloat16* VnT;    // [nblk, H, dv, BT]      V^new^T             (backward)
  __nv_bfloat16* dHT;    // [nblk, H, dv, 128]     dH_{b+1}^T          (backward)
  __nv_bfloat16* dVnT;   // [nblk, H, dv, BT]      dV^new^T            (backward)
  float* Sseg[2];        // [B, H, dk, dv] x 2     fp32 state between the segments of a split forward
};

// How a fixed-length forward call is carried out: nseg = 1 runs Pre over
// the whole chunk, then the chain; nseg > 1 splits the chunk's blocks at
// b[1..nseg-1] (64-token boundaries) and overlaps Pre of one segment with the
// chain of the previous one. chain_rg = value-row groups of 16 per chain CTA.
struct FwdSplit {
  static constexpr int kMaxSeg = 16;
  int nseg = 1;
  int chain_rg = 1;
  int b[kMaxSeg + 1] = {};
};

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

}  // namespace gdn
