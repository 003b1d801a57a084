// The sequential state chains of the bf16 tensor-core path (the ST step of the
// StateFlow review's Pre / ST / Out decomposition, Eq. 2, and its reverse for
// the backward pass, Eq. 6-7), plus the orchestration of the forward and
// backward calls.
//
// One CTA carries RG x 16 value columns of one (sequence, head) through the
// sequence's 64-token blocks in order: 4 compute warps and one producer warp.
// The producer fills a ring of stages with bulk copies of the block's operand
// tiles (written by Pre with padded rows), tracked by mbarriers; the compute
// warps keep the fp32 state in registers and use warp-level bf16 MMAs.
// Compute warp w owns key columns [32w, 32w + 32) of the state and tokens
// [16w, 16w + 16) of each block.
//
// Pre hands over the decay-scaled copies K~ = diag(e^{gamma_C - gamma}) K and
// Q~ = diag(e^{gamma}) Q, so every decay factor of a step except Gamma_C sits
// in an operand. Forward chain, per block (H^T: value rows x key columns):
//   X^T    = H^T W^T ;  V^new^T = U^T - X^T
//   H^T   <- Gamma_C H^T + V^new^T K~
//   O^T    = H^T Q~^T + V^new^T QKM^T                   (forward mode only)
// Reverse chain, per block from the last one (dH = dS_out at the start):
//   dV^new = QKM^T dO + K~ dH ;  dH <- Gamma_C dH + Q~^T dO - W^T dV^new
// The backward call runs the recompute chain (which rebuilds H_b and V^new
// from S_in) and the reverse chain concurrently: they depend only on Pre.
#include <cstddef>
#include <mutex>

#include "gdn_internal.cuh"
#include "gdn_mma.cuh"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

constexpr int LDK = TC_LDK;
constexpr int LD64 = TC_LD64;
constexpr int LDU = TC_LDU;
constexpr int DK = 128;
constexpr int CHAIN_THREADS = 160;  // 4 compute warps + 1 producer warp

enum { CHAIN_FWD = 0, CHAIN_RECOMPUTE = 1 };

// Internal streams of the split forward (created once per device): Pre on
// the lowest priority, the chain on the highest, so the chain's CTAs take
// SMs first and Pre fills the rest. Calls that split share them: the host
// side of a split call holds the device's lock while it enqueues.
struct SideStreams {
  std::mutex mu;
  cudaStream_t pre = nullptr, chain = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, seg[FwdSplit::kMaxSeg] = {};
};

SideStreams* side_streams() {
  static std::mutex init_mu;
  static SideStreams* per_dev[64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(init_mu);
  if (!per_dev[dev]) {
    SideStreams* ss = new SideStreams();
    int least = 0, greatest = 0;
    bool ok = cudaDeviceGetStreamPriorityRange(&least, &greatest) == cudaSuccess &&
              cudaStreamCreateWithPriority(&ss->pre, cudaStreamNonBlocking, least) == cudaSuccess &&
              cudaStreamCreateWithPriority(&ss->chain, cudaStreamNonBlocking, greatest) == cudaSuccess &&
              cudaEventCreateWithFlags(&ss->fork, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&ss->join, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < FwdSplit::kMaxSeg; ++i)
      ok = cudaEventCreateWithFlags(&ss->seg[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return nullptr;  // (the handles stay with the process; no call uses them)
    per_dev[dev] = ss;
  }
  return per_dev[dev];
}

// Fragment loads of mma.m16n8k16 from a 128-byte-swizzled tile (64-wide column
// tiles `tb` bytes apart; sw128 of gdn_umma.cuh), with the lane -> (row,
// column) assignment of ldb_nk_x2n and ldb_kn_x2n. Q~ and QKM arrive in this
// layout.
__device__ __forceinline__ void ldb_nk_sw(uint32_t* b, uint32_t base, uint32_t tb, int n0, int k0) {
  const int l = threadIdx.x & 31, mat = l >> 3;
  ldsm_x4(base + sw128(n0 + (l & 7) + (mat >> 1) * 8, k0 + (mat & 1) * 8, tb), b[0], b[1], b[2], b[3]);
}
__device__ __forceinline__ void ldb_kn_sw(uint32_t* b, uint32_t base, uint32_t tb, int k0, int n0) {
  const int l = threadIdx.x & 31, mat = l >> 3;
  ldsm_x4_t(base + sw128(k0 + (l & 7) + (mat & 1) * 8, n0 + (mat >> 1) * 8, tb), b[0], b[1], b[2],
            b[3]);
}

// ------------------------------------------------------------------ forward / recompute
template <int MODE, int RG>
struct FwdStage {
  __nv_bfloat16 W[2 * BT * 64];  // swizzled [t][64 key] tiles
  __nv_bfloat16 K[2 * BT * 64];  // swizzled [t][64 key] tiles
  __nv_bfloat16 Q[MODE == CHAIN_FWD ? 2 * BT * 64 : 8];  // swizzled [t][64 key] tiles
  __nv_bfloat16 QKM[MODE == CHAIN_FWD ? BT * 64 : 8];    // swizzled [t][j] tile
  __nv_bfloat16 U[RG * BT * LDU];
  float dec[3 * BT];
};

template <int MODE, int RG>
constexpr int fwd_stages() {
  return MODE == CHAIN_FWD ? 3 : 4;
}

template <int MODE, int RG>
struct FwdSmem {
  FwdStage<MODE, RG> st[fwd_stages<MODE, RG>()];
  uint64_t full[fwd_stages<MODE, RG>()];
  uint64_t empty[fwd_stages<MODE, RG>()];
  __nv_bfloat16 HT[16 * RG * LDK];
  __nv_bfloat16 VnT[16 * RG * LD64];
  __nv_bfloat16 O[MODE == CHAIN_FWD ? BT * (16 * RG + 8) : 8];
  int abort;
};
using FwdStage2 = FwdStage<CHAIN_FWD, 2>;
static_assert(sizeof(FwdStage<CHAIN_FWD, 1>) % 16 == 0 && sizeof(FwdStage2) % 16 == 0 &&
                  sizeof(FwdStage<CHAIN_RECOMPUTE, 2>) % 16 == 0 && offsetof(FwdStage2, Q) % 16 == 0 &&
                  offsetof(FwdStage2, QKM) % 16 == 0 && offsetof(FwdStage2, U) % 16 == 0 &&
                  offsetof(FwdStage2, dec) % 16 == 0,
              "chain copy destinations start on 16 bytes");

// Blocks [lb0, min(lb1, nblk)) of each sequence: the whole sequence, or one
// segment of a split forward call (the state enters from S_in and leaves
// through S_out, both exact fp32).
template <int DV, int MODE, int RG>
__device__ __forceinline__ void chain_fwd_body(const SeqMap& m, int cta,
                                               const __nv_bfloat16* __restrict__ q,
                                               const __nv_bfloat16* __restrict__ k,
                                               const float* S_in, float* S_out,
                                               __nv_bfloat16* __restrict__ o, const TcWs& ws,
                                               unsigned char* smraw, int lb0 = 0,
                                               int lb1 = 1 << 30) {
  constexpr int BV = 16 * RG;
  constexpr int NVT = DV / BV;
  constexpr int NS = fwd_stages<MODE, RG>();
  constexpr int LDO = BV + 8;
  const int tile = cta % NVT;
  const int sh = cta / NVT;
  const int H = m.H, h = sh % H, s = m.order ? m.order[sh / H] : sh / H;
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31, gq = l >> 2, tq = l & 3;
  const SeqInfo si = seq_info(m, s);
  const int nb = max(0, min(si.nblk, lb1) - lb0);  // blocks this launch carries
  FwdSmem<MODE, RG>& sm = *reinterpret_cast<FwdSmem<MODE, RG>*>(smraw);
  volatile int* abort = &sm.abort;
  // H_b and V^new of every block go to the workspace for the gradient kernel:
  // always when recomputing, and from the forward when the caller keeps them
  const bool keep = MODE == CHAIN_RECOMPUTE || ws.HbT != nullptr;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 4);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  const size_t sbase = ((size_t)s * H + h) * DK * DV + (size_t)tile * BV;
  // fp32 state slices: row group g holds H^T rows v = 16g + gq (+8), key columns 32w + 8j + 2tq (+1)
  float hs[RG][4][4];
  if (w < 4) {
#pragma unroll
    for (int g = 0; g < RG; ++g)
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int vr = 16 * g + gq + 8 * (e >> 1);
          const int kc = 32 * w + 8 * j + 2 * tq + (e & 1);
          hs[g][j][e] = S_in ? S_in[sbase + (size_t)kc * DV + vr] : 0.f;
        }
#pragma unroll
    for (int g = 0; g < RG; ++g)
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int vr = 16 * g + gq + 8 * hf, kc = 32 * w + 8 * j + 2 * tq;
          *reinterpret_cast<uint32_t*>(&sm.HT[vr * LDK + kc]) =
              pack_bf16(hs[g][j][2 * hf], hs[g][j][2 * hf + 1]);
        }
  }
  __syncthreads();

  if (w == 4) {
    // ---------------- producer warp
    int issued = 0;
    for (int i = 0; i < nb; ++i) {
      const int lb = lb0 + i;
      const int st = i % NS, kf = i / NS;
      if (i >= NS && !mbar_wait(&sm.empty[st], (kf - 1) & 1, abort)) break;
      FwdStage<MODE, RG>& S = sm.st[st];
      const size_t bh = (size_t)(si.blk0 + lb) * H + h;
      const uint32_t bytes = 4 * BT * 64 * 2 + RG * BT * LDU * 2 + 3 * BT * 4 +
                             (MODE == CHAIN_FWD ? 3 * BT * 64 * 2 : 0);
      if (l == 0) {
        uint64_t* fb = &sm.full[st];
        mbar_arrive_expect_tx(fb, bytes);
        bulk_g2s(S.W, ws.W + bh * BT * LDK, 2 * BT * 64 * 2, fb);
        bulk_g2s(S.K, ws.Kp + bh * BT * LDK, 2 * BT * 64 * 2, fb);
        bulk_g2s(S.dec, ws.dec + bh * TC_DEC_ROWS * BT, 3 * BT * 4, fb);
        bulk_g2s(S.U, ws.U + (bh * (DV / 16) + (size_t)tile * RG) * BT * LDU, RG * BT * LDU * 2, fb);
        if (MODE == CHAIN_FWD) {
          bulk_g2s(S.Q, ws.Qp + bh * BT * LDK, 2 * BT * 64 * 2, fb);
          bulk_g2s(S.QKM, ws.QKM + bh * BT * LD64, BT * 64 * 2, fb);
        }
      }
      ++issued;
    }
    __syncwarp();
    if (*abort && l == 0) {  // after a timeout: let every copy still in flight land
      for (int i = max(0, issued - NS); i < issued; ++i) {
        const long long t0 = clock64();
        while (!mbar_try_wait(&sm.full[i % NS], (i / NS) & 1) && clock64() - t0 < (1ll << 31)) {
        }
      }
    }
  } else {
    // ---------------- compute warps
    for (int i = 0; i < nb; ++i) {
      const int lb = lb0 + i;
      const int st = i % NS;
      const bool ok = mbar_wait(&sm.full[st], (i / NS) & 1, abort);
      const FwdStage<MODE, RG>& S = sm.st[st];
      const int tok0 = si.tok0 + lb * BT, len = min(BT, si.len - lb * BT);
      const size_t bh = (size_t)(si.blk0 + lb) * H + h;
      const float* dec = S.dec;
      // X^T = H^T W^T (W fragments shared by the row groups) and, forward, H^T Q~^T
      // from the same H^T fragments
      float x[RG][2][2][4], o1[RG][2][2][4];
#pragma unroll
      for (int g = 0; g < RG; ++g)
#pragma unroll
        for (int p = 0; p < 2; ++p)
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) x[g][p][j][e] = o1[g][p][j][e] = 0.f;
      {
        uint32_t bW[DK / 16][4];
#pragma unroll
        for (int kc = 0; kc < DK / 16; ++kc) ldb_nk_sw(bW[kc], smem_u32(S.W), 8192, 16 * w, 16 * kc);
#pragma unroll
        for (int g = 0; g < RG; ++g) {
          uint32_t aH[DK / 16][4];
#pragma unroll
          for (int kc = 0; kc < DK / 16; ++kc) lda_rm(aH[kc], sm.HT, LDK, 16 * g, 16 * kc);
#pragma unroll
          for (int kc = 0; kc < DK / 16; ++kc) {
            mma16816(x[g][kc & 1][0], aH[kc], bW[kc][0], bW[kc][1]);
            mma16816(x[g][kc & 1][1], aH[kc], bW[kc][2], bW[kc][3]);
          }
          if (MODE == CHAIN_FWD) {
#pragma unroll
            for (int kc = 0; kc < DK / 16; ++kc) {
              uint32_t bQ[4];
              ldb_nk_sw(bQ, smem_u32(S.Q), 8192, 16 * w, 16 * kc);
              mma16816(o1[g][kc & 1][0], aH[kc], bQ[0], bQ[1]);
              mma16816(o1[g][kc & 1][1], aH[kc], bQ[2], bQ[3]);
            }
          }
        }
      }
      // H_b for the gradient kernel (after the MMAs that read H^T were issued;
      // H^T is rewritten only after the next barrier)
      if (keep && ok) {
        __nv_bfloat16* Hg = ws.HbT + bh * DV * DK + (size_t)tile * BV * DK;
        for (int idx = tid; idx < BV * 16; idx += 128) {
          const int r = idx >> 4, c = (idx & 15) * 8;
          *reinterpret_cast<uint4*>(Hg + r * DK + c) =
              *reinterpret_cast<const uint4*>(&sm.HT[r * LDK + c]);
        }
      }
      // V^new^T = U^T - X^T (the forward keeps it in registers too and writes
      // its global copy once the next phase's MMAs are issued)
      uint32_t pvs[RG][2][2];
#pragma unroll
      for (int g = 0; g < RG; ++g) {
        // U^T fragments at the accumulator positions (value rows, token pairs):
        // a transposing matrix load of the token-major U tile, matrix 2j + hf
        // = tokens [16w + 8j, +8) x values [8hf, +8)
        uint32_t uf[4];
        {
          const int mi = l >> 3;
          ldsm_x4_t(smem_u32(S.U + g * BT * LDU + u_tile_off(16 * w + 8 * (mi >> 1) + (l & 7), 8 * (mi & 1))),
                    uf[0], uf[1], uf[2], uf[3]);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int vr = 16 * g + gq + 8 * hf;
            const int t0 = 16 * w + 8 * j + 2 * tq;
            const float2 uu = unpack_bf16(uf[2 * j + hf]);
            const float u0 = uu.x, u1 = uu.y;
            const float v0 = u0 - (x[g][0][j][2 * hf] + x[g][1][j][2 * hf]);
            const float v1 = u1 - (x[g][0][j][2 * hf + 1] + x[g][1][j][2 * hf + 1]);
            const uint32_t pv = pack_bf16(v0, v1);
            *reinterpret_cast<uint32_t*>(&sm.VnT[vr * LD64 + t0]) = pv;
            if (MODE == CHAIN_FWD)
              pvs[g][j][hf] = pv;
            else if (ok)
              *reinterpret_cast<uint32_t*>(ws.VnT + bh * DV * BT + (size_t)(tile * BV + vr) * BT + t0) = pv;
          }
      }
      // operands of the state update that do not depend on V^new: load before the barrier
      uint32_t bK[4][8], bM[4][4];
#pragma unroll
      for (int kc = 0; kc < 4; ++kc) {
        ldb_kn_sw(&bK[kc][0], smem_u32(S.K), 8192, 16 * kc, 32 * w);
        ldb_kn_sw(&bK[kc][4], smem_u32(S.K), 8192, 16 * kc, 32 * w + 16);
        if (MODE == CHAIN_FWD) ldb_nk_sw(bM[kc], smem_u32(S.QKM), 0, 16 * w, 16 * kc);
      }
      named_bar(1, 128);

      // H^T <- Gamma_C H^T + V^new^T K~ on key columns [32w, 32w + 32); forward:
      // O^T = H_b^T Q~^T + V^new^T QKM^T from the same V^new^T fragments
      const float GC = dec[BT - 1];
#pragma unroll
      for (int g = 0; g < RG; ++g) {
        float h2[4][4], o2[2][4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hs[g][j][e] *= GC;
            h2[j][e] = 0.f;
          }
        uint32_t aV[4][4];
#pragma unroll
        for (int kc = 0; kc < 4; ++kc) lda_rm(aV[kc], sm.VnT, LD64, 16 * g, 16 * kc);
#pragma unroll
        for (int kc = 0; kc < 4; ++kc) {
          float(*acc)[4] = (kc & 1) ? h2 : hs[g];
#pragma unroll
          for (int j = 0; j < 4; ++j) mma16816(acc[j], aV[kc], bK[kc][2 * j], bK[kc][2 * j + 1]);
        }
        if (MODE == CHAIN_FWD && keep && ok) {
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
              *reinterpret_cast<uint32_t*>(ws.VnT + bh * DV * BT +
                                           (size_t)(tile * BV + 16 * g + gq + 8 * hf) * BT +
                                           16 * w + 8 * j + 2 * tq) = pvs[g][j][hf];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) hs[g][j][e] += h2[j][e];
        if (MODE == CHAIN_FWD) {
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) o2[j][e] = o1[g][0][j][e] + o1[g][1][j][e];
#pragma unroll
          for (int kc = 0; kc < 4; ++kc) {
            mma16816(o2[0], aV[kc], bM[kc][0], bM[kc][1]);
            mma16816(o2[1], aV[kc], bM[kc][2], bM[kc][3]);
          }
          // O[token][v]: the transposing matrix store turns the (value, token)
          // fragments into token rows for coalesced global stores
          const int mi = l >> 3;
          stsm_x4_t(smem_u32(&sm.O[(16 * w + 8 * (mi >> 1) + (l & 7)) * LDO + 16 * g + 8 * (mi & 1)]),
                    pack_bf16(o2[0][0], o2[0][1]), pack_bf16(o2[0][2], o2[0][3]),
                    pack_bf16(o2[1][0], o2[1][1]), pack_bf16(o2[1][2], o2[1][3]));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int vr = 16 * g + gq + 8 * hf, kc = 32 * w + 8 * j + 2 * tq;
            *reinterpret_cast<uint32_t*>(&sm.HT[vr * LDK + kc]) =
                pack_bf16(hs[g][j][2 * hf], hs[g][j][2 * hf + 1]);
          }
      }
      if (MODE == CHAIN_FWD) {
        __syncwarp();
        // each warp stores its own 16 tokens: BV / 8 chunks of 16 bytes per row
        for (int idx = l; idx < 16 * (BV / 8); idx += 32) {
          const int r = 16 * w + idx / (BV / 8), c = (idx % (BV / 8)) * 8;
          if (r < len && ok)
            *reinterpret_cast<uint4*>(o + ((size_t)(tok0 + r) * H + h) * DV + tile * BV + c) =
                *reinterpret_cast<const uint4*>(&sm.O[r * LDO + c]);
        }
      }
      __syncwarp();
      if (l == 0) mbar_arrive(&sm.empty[st]);
      named_bar(1, 128);
    }
    if (S_out && !*abort) {
#pragma unroll
      for (int g = 0; g < RG; ++g)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int vr = 16 * g + gq + 8 * (e >> 1);
            const int kc = 32 * w + 8 * j + 2 * tq + (e & 1);
            S_out[sbase + (size_t)kc * DV + vr] = hs[g][j][e];
          }
    }
  }
  __syncthreads();
  if (tid == 0 && *abort) ws.status[0] = DEV_TIMEOUT;
}

// ------------------------------------------------------------------ reverse chain
template <int RG>
struct RevStage {
  __nv_bfloat16 W[2 * BT * 64];  // swizzled [t][64 key] tiles
  __nv_bfloat16 K[2 * BT * 64];  // swizzled [t][64 key] tiles
  __nv_bfloat16 Q[2 * BT * 64];  // swizzled [t][64 key] tiles
  __nv_bfloat16 QKM[BT * 64];    // swizzled [t][j] tile
  __nv_bfloat16 dO[BT * (16 * RG + 8)];
  float dec[3 * BT];
};

constexpr int REV_STAGES = 3;

template <int RG>
struct RevSmem {
  RevStage<RG> st[REV_STAGES];
  uint64_t full[REV_STAGES];
  uint64_t empty[REV_STAGES];
  __nv_bfloat16 dHT[16 * RG * LDK];   // bf16 copy of dH^T (value rows)
  __nv_bfloat16 dVT[16 * RG * LD64];  // -dV^new^T (value rows)
  int abort;
};
static_assert(sizeof(RevStage<1>) % 16 == 0 && sizeof(RevStage<2>) % 16 == 0 &&
                  offsetof(RevStage<2>, Q) % 16 == 0 && offsetof(RevStage<2>, QKM) % 16 == 0 &&
                  offsetof(RevStage<2>, dO) % 16 == 0 && offsetof(RevStage<2>, dec) % 16 == 0,
              "reverse-chain copy destinations start on 16 bytes");

template <int DV, int RG>
__device__ __forceinline__ void chain_rev_body(const SeqMap& m, int cta,
                                               const __nv_bfloat16* __restrict__ q,
                                               const __nv_bfloat16* __restrict__ k,
                                               const __nv_bfloat16* __restrict__ dout,
                                               const float* dS_out, float* dS_in, const TcWs& ws,
                                               unsigned char* smraw) {
  constexpr int BV = 16 * RG;
  constexpr int NVT = DV / BV;
  constexpr int NS = REV_STAGES;
  constexpr int LDO = BV + 8;
  const int tile = cta % NVT;
  const int sh = cta / NVT;
  const int H = m.H, h = sh % H, s = m.order ? m.order[sh / H] : sh / H;
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31, gq = l >> 2, tq = l & 3;
  const SeqInfo si = seq_info(m, s);
  RevSmem<RG>& sm = *reinterpret_cast<RevSmem<RG>*>(smraw);
  volatile int* abort = &sm.abort;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sm.full[i], 1 + 32);  // bulk-copy arrival + one cp.async arrival per producer lane
      mbar_init(&sm.empty[i], 4);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  float dh[RG][4][4];
  const size_t sbase = ((size_t)s * H + h) * DK * DV + (size_t)tile * BV;
  if (w < 4) {
#pragma unroll
    for (int g = 0; g < RG; ++g)
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int vr = 16 * g + gq + 8 * (e >> 1);
          const int kc = 32 * w + 8 * j + 2 * tq + (e & 1);
          dh[g][j][e] = dS_out ? dS_out[sbase + (size_t)kc * DV + vr] : 0.f;
        }
#pragma unroll
    for (int g = 0; g < RG; ++g)
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int vr = 16 * g + gq + 8 * hf, kc = 32 * w + 8 * j + 2 * tq;
          *reinterpret_cast<uint32_t*>(&sm.dHT[vr * LDK + kc]) =
              pack_bf16(dh[g][j][2 * hf], dh[g][j][2 * hf + 1]);
        }
  }
  __syncthreads();

  if (w == 4) {
    // ---------------- producer warp: iteration it loads block nblk - 1 - it
    int issued = 0;
    for (int it = 0; it < si.nblk; ++it) {
      const int st = it % NS, kf = it / NS;
      if (it >= NS && !mbar_wait(&sm.empty[st], (kf - 1) & 1, abort)) break;
      RevStage<RG>& S = sm.st[st];
      const int lb = si.nblk - 1 - it;
      const int tok0 = si.tok0 + lb * BT, len = min(BT, si.len - lb * BT);
      const size_t bh = (size_t)(si.blk0 + lb) * H + h;
      const uint32_t bytes = 7 * BT * 64 * 2 + 3 * BT * 4;
      if (l == 0) {
        uint64_t* fb = &sm.full[st];
        mbar_arrive_expect_tx(fb, bytes);
        bulk_g2s(S.W, ws.W + bh * BT * LDK, 2 * BT * 64 * 2, fb);
        bulk_g2s(S.K, ws.Kp + bh * BT * LDK, 2 * BT * 64 * 2, fb);
        bulk_g2s(S.Q, ws.Qp + bh * BT * LDK, 2 * BT * 64 * 2, fb);
        bulk_g2s(S.QKM, ws.QKM + bh * BT * LD64, BT * 64 * 2, fb);
        bulk_g2s(S.dec, ws.dec + bh * TC_DEC_ROWS * BT, 3 * BT * 4, fb);
      }
      // the dO tile: 16-byte cp.async per lane, rows past the block's end zero-filled
#pragma unroll
      for (int idx = l; idx < BT * (BV / 8); idx += 32) {
        const int r = idx / (BV / 8), c = (idx % (BV / 8)) * 8;
        const bool okr = r < len;
        const size_t tok = (size_t)(tok0 + (okr ? r : 0)) * H + h;
        cp16(&S.dO[r * LDO + c], dout + tok * DV + tile * BV + c, okr);
      }
      cp_async_mbar_arrive(&sm.full[st]);
      ++issued;
    }
    cp_wait<0>();
    __syncwarp();
    if (*abort && l == 0) {
      for (int it = max(0, issued - NS); it < issued; ++it) {
        const long long t0 = clock64();
        while (!mbar_try_wait(&sm.full[it % NS], (it / NS) & 1) && clock64() - t0 < (1ll << 31)) {
        }
      }
    }
  } else {
    // ---------------- compute warps
    for (int it = 0; it < si.nblk; ++it) {
      const int st = it % NS;
      const bool ok = mbar_wait(&sm.full[st], (it / NS) & 1, abort);
      const RevStage<RG>& S = sm.st[st];
      const int lb = si.nblk - 1 - it;
      const size_t bh = (size_t)(si.blk0 + lb) * H + h;
      const float* dec = S.dec;
      // dV^new^T for tokens [16w, 16w + 16): dO^T QKM + dH^T K~^T; the dO^T
      // fragments are kept for the dH update
      uint32_t aO[RG][4][4];
      {
        uint32_t bK[DK / 16][4], bM[4][4];
#pragma unroll
        for (int kc = 0; kc < DK / 16; ++kc) ldb_nk_sw(bK[kc], smem_u32(S.K), 8192, 16 * w, 16 * kc);
#pragma unroll
        for (int kc = 0; kc < 4; ++kc) ldb_kn_sw(bM[kc], smem_u32(S.QKM), 0, 16 * kc, 16 * w);
#pragma unroll
        for (int g = 0; g < RG; ++g) {
          float a1[2][4], a2[2][2][4];
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) a1[j][e] = a2[0][j][e] = a2[1][j][e] = 0.f;
          uint32_t aD[DK / 16][4];
#pragma unroll
          for (int kc = 0; kc < DK / 16; ++kc) lda_rm(aD[kc], sm.dHT, LDK, 16 * g, 16 * kc);
#pragma unroll
          for (int kc = 0; kc < DK / 16; ++kc) {
            mma16816(a2[kc & 1][0], aD[kc], bK[kc][0], bK[kc][1]);
            mma16816(a2[kc & 1][1], aD[kc], bK[kc][2], bK[kc][3]);
          }
#pragma unroll
          for (int kc = 0; kc < 4; ++kc) lda_tr(aO[g][kc], S.dO, LDO, 16 * g, 16 * kc);
#pragma unroll
          for (int kc = 0; kc < 4; ++kc) {
            mma16816(a1[0], aO[g][kc], bM[kc][0], bM[kc][1]);
            mma16816(a1[1], aO[g][kc], bM[kc][2], bM[kc][3]);
          }
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int vr = 16 * g + gq + 8 * hf;
              const int t0 = 16 * w + 8 * j + 2 * tq;
              const float d0 = a1[j][2 * hf] + (a2[0][j][2 * hf] + a2[1][j][2 * hf]);
              const float d1 = a1[j][2 * hf + 1] + (a2[0][j][2 * hf + 1] + a2[1][j][2 * hf + 1]);
              *reinterpret_cast<uint32_t*>(&sm.dVT[vr * LD64 + t0]) = pack_bf16(-d0, -d1);
              if (ok)
                *reinterpret_cast<uint32_t*>(ws.dVnT + bh * DV * BT + (size_t)(tile * BV + vr) * BT + t0) =
                    pack_bf16(d0, d1);
            }
        }
      }
      // dH_{b+1} (bf16, value-major) for the gradient kernel (dH^T is rewritten
      // only after the next barrier)
      if (ok) {
        __nv_bfloat16* Dg = ws.dHT + bh * DV * DK + (size_t)tile * BV * DK;
        for (int idx = tid; idx < BV * 16; idx += 128) {
          const int r = idx >> 4, c = (idx & 15) * 8;
          *reinterpret_cast<uint4*>(Dg + r * DK + c) =
              *reinterpret_cast<const uint4*>(&sm.dHT[r * LDK + c]);
        }
      }
      // operands that do not depend on dV^new: load before the barrier
      uint32_t bQ[4][8], bW[4][8];
#pragma unroll
      for (int kc = 0; kc < 4; ++kc) {
        ldb_kn_sw(&bQ[kc][0], smem_u32(S.Q), 8192, 16 * kc, 32 * w);
        ldb_kn_sw(&bQ[kc][4], smem_u32(S.Q), 8192, 16 * kc, 32 * w + 16);
        ldb_kn_sw(&bW[kc][0], smem_u32(S.W), 8192, 16 * kc, 32 * w);
        ldb_kn_sw(&bW[kc][4], smem_u32(S.W), 8192, 16 * kc, 32 * w + 16);
      }
      named_bar(1, 128);
      // dH^T <- Gamma_C dH^T + dO^T Q~ - dV^new^T W on key columns [32w, 32w + 32)
      const float GC = dec[BT - 1];
#pragma unroll
      for (int g = 0; g < RG; ++g) {
        float d2[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dh[g][j][e] *= GC;
            d2[j][e] = 0.f;
          }
        uint32_t aV[4][4];
#pragma unroll
        for (int kc = 0; kc < 4; ++kc) lda_rm(aV[kc], sm.dVT, LD64, 16 * g, 16 * kc);
#pragma unroll
        for (int kc = 0; kc < 4; ++kc) {
#pragma unroll
          for (int j = 0; j < 4; ++j) mma16816(dh[g][j], aO[g][kc], bQ[kc][2 * j], bQ[kc][2 * j + 1]);
#pragma unroll
          for (int j = 0; j < 4; ++j) mma16816(d2[j], aV[kc], bW[kc][2 * j], bW[kc][2 * j + 1]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) dh[g][j][e] += d2[j][e];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int vr = 16 * g + gq + 8 * hf, kc = 32 * w + 8 * j + 2 * tq;
            *reinterpret_cast<uint32_t*>(&sm.dHT[vr * LDK + kc]) =
                pack_bf16(dh[g][j][2 * hf], dh[g][j][2 * hf + 1]);
          }
      }
      __syncwarp();
      if (l == 0) mbar_arrive(&sm.empty[st]);
      named_bar(1, 128);
    }
    if (dS_in && !*abort) {
#pragma unroll
      for (int g = 0; g < RG; ++g)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int vr = 16 * g + gq + 8 * (e >> 1);
            const int kc = 32 * w + 8 * j + 2 * tq + (e & 1);
            dS_in[sbase + (size_t)kc * DV + vr] = dh[g][j][e];
          }
    }
  }
  __syncthreads();
  if (tid == 0 && *abort) ws.status[0] = DEV_TIMEOUT;
}

// ------------------------------------------------------------------ kernels
// Forward: 16 value columns per CTA (the most SMs per head: the chain step is
// bounded by each CTA's shared-memory traffic, which does not shrink with fewer
// columns per CTA).
template <int DV, int RG>
__global__ void __launch_bounds__(CHAIN_THREADS, 1)
    k_chain_fwd(SeqMap m, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                const float* S_in, float* S_out, __nv_bfloat16* __restrict__ o, TcWs ws, int lb0,
                int lb1) {
  extern __shared__ __align__(128) unsigned char smraw[];
  chain_fwd_body<DV, CHAIN_FWD, RG>(m, blockIdx.x, q, k, S_in, S_out, o, ws, smraw, lb0, lb1);
}

// Backward: the recompute chain (CTAs [0, n)) and the reverse chain (CTAs
// [n, 2n)) run side by side, 32 value columns per CTA.
constexpr int BWD_RG = 2;

template <int DV>
__global__ void __launch_bounds__(CHAIN_THREADS, 1)
    k_chains_bwd(SeqMap m, int n, const __nv_bfloat16* __restrict__ q,
                 const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ dout,
                 const float* S_in, const float* dS_out, float* dS_in, TcWs ws) {
  extern __shared__ __align__(128) unsigned char smraw[];
  if ((int)blockIdx.x < n)
    chain_fwd_body<DV, CHAIN_RECOMPUTE, BWD_RG>(m, blockIdx.x, q, k, S_in, nullptr, nullptr, ws,
                                               smraw);
  else
    chain_rev_body<DV, BWD_RG>(m, blockIdx.x - n, q, k, dout, dS_out, dS_in, ws, smraw);
}

// Backward from kept forward products: H_b and V^new are already in the
// workspace, so only the reverse chain runs, 16 value columns per CTA.
template <int DV>
__global__ void __launch_bounds__(CHAIN_THREADS, 1)
    k_chain_rev(SeqMap m, const __nv_bfloat16* __restrict__ q,
                const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ dout,
                const float* dS_out, float* dS_in, TcWs ws) {
  extern __shared__ __align__(128) unsigned char smraw[];
  chain_rev_body<DV, 1>(m, blockIdx.x, q, k, dout, dS_out, dS_in, ws, smraw);
}

template <class K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int DV, int RG>
cudaError_t launch_chain_fwd(const SeqMap& m, const void* q, const void* k, const float* S_in,
                             void* o, float* S_out, const TcWs& ws, int lb0, int lb1,
                             cudaStream_t st, bool mark) {
  using bf = __nv_bfloat16;
  constexpr size_t smem = sizeof(FwdSmem<CHAIN_FWD, RG>);
  cudaError_t e;
  if ((e = set_smem(k_chain_fwd<DV, RG>, smem))) return e;
  if (mark) prof_mark(st, ws.HbT ? "tc_chain_fwd_keep" : "tc_chain_fwd");
  k_chain_fwd<DV, RG><<<m.nseq * m.H * (DV / (16 * RG)), CHAIN_THREADS, smem, st>>>(
      m, (const bf*)q, (const bf*)k, S_in, S_out, (bf*)o, ws, lb0, lb1);
  return cudaGetLastError();
}

template <int DV>
cudaError_t fwd_t(const SeqMap& m, const void* q, const void* k, const void* v, const void* g,
                  const void* beta, const float* S_in, void* o, float* S_out, const TcWs& ws,
                  const FwdSplit& sp, cudaStream_t st) {
  cudaError_t e;
  if (sp.nseg <= 1) {
    if ((e = tc_pre(m, DV, q, k, v, g, beta, ws, 0, 0, st, true))) return e;
    e = sp.chain_rg == 2 ? launch_chain_fwd<DV, 2>(m, q, k, S_in, o, S_out, ws, 0, 1 << 30, st, true)
                         : launch_chain_fwd<DV, 1>(m, q, k, S_in, o, S_out, ws, 0, 1 << 30, st, true);
    prof_mark(st, nullptr);
    return e;
  }
  // State-transition / dense-kernel overlap: Pre of segment i + 1 on a
  // low-priority stream while the chain carries segment i on a high-priority
  // one; the chain's fp32 state passes between segments through the
  // workspace exactly, so the results equal the unsplit call's bit for bit.
  SideStreams* ss = side_streams();
  if (!ss) return cudaErrorUnknown;
  std::lock_guard<std::mutex> lock(ss->mu);
  prof_mark(st, "tc_fwd_overlap");
  if ((e = cudaEventRecord(ss->fork, st)) || (e = cudaStreamWaitEvent(ss->pre, ss->fork, 0)) ||
      (e = cudaStreamWaitEvent(ss->chain, ss->fork, 0)))
    return e;
  for (int i = 0; i < sp.nseg; ++i) {
    const int b0 = sp.b[i], b1 = sp.b[i + 1];
    if ((e = tc_pre(m, DV, q, k, v, g, beta, ws, b0, b1 - b0, ss->pre, false))) return e;
    if ((e = cudaEventRecord(ss->seg[i], ss->pre))) return e;
  }
  for (int i = 0; i < sp.nseg; ++i) {
    const float* sin = i == 0 ? S_in : ws.Sseg[(i - 1) & 1];
    float* sout = i == sp.nseg - 1 ? S_out : ws.Sseg[i & 1];
    if ((e = cudaStreamWaitEvent(ss->chain, ss->seg[i], 0))) return e;
    e = sp.chain_rg == 2
            ? launch_chain_fwd<DV, 2>(m, q, k, sin, o, sout, ws, sp.b[i], sp.b[i + 1], ss->chain, false)
            : launch_chain_fwd<DV, 1>(m, q, k, sin, o, sout, ws, sp.b[i], sp.b[i + 1], ss->chain, false);
    if (e) return e;
  }
  if ((e = cudaEventRecord(ss->join, ss->chain)) || (e = cudaStreamWaitEvent(st, ss->join, 0)))
    return e;
  prof_mark(st, nullptr);
  return cudaSuccess;
}

template <int DV>
cudaError_t bwd_t(const SeqMap& m, const void* q, const void* k, const void* v, const void* g,
                  const void* beta, const float* S_in, const void* dout, const float* dS_out,
                  void* dq, void* dkk, void* dvv, void* dg, void* dbeta, float* dS_in,
                  const TcWs& ws, bool run_pre, cudaStream_t st) {
  using bf = __nv_bfloat16;
  cudaError_t e;
  if (!run_pre) {
    // H_b, V^new and the Pre products come from the forward call
    constexpr size_t smem = sizeof(RevSmem<1>);
    if ((e = set_smem(k_chain_rev<DV>, smem))) return e;
    prof_mark(st, "tc_chain_rev");
    k_chain_rev<DV><<<m.nseq * m.H * (DV / 16), CHAIN_THREADS, smem, st>>>(
        m, (const bf*)q, (const bf*)k, (const bf*)dout, dS_out, dS_in, ws);
    if ((e = cudaGetLastError())) return e;
    if ((e = tc_grad(m, DV, q, k, v, beta, dout, dq, dkk, dvv, dg, dbeta, ws, st))) return e;
    prof_mark(st, nullptr);
    return cudaGetLastError();
  }
  if ((e = tc_pre(m, DV, q, k, v, g, beta, ws, 0, 0, st, true))) return e;
  constexpr size_t s1 = sizeof(FwdSmem<CHAIN_RECOMPUTE, BWD_RG>);
  constexpr size_t s2 = sizeof(RevSmem<BWD_RG>);
  constexpr size_t smem = s1 > s2 ? s1 : s2;
  if ((e = set_smem(k_chains_bwd<DV>, smem))) return e;
  const int n = m.nseq * m.H * (DV / (16 * BWD_RG));
  prof_mark(st, "tc_chains_bwd");
  k_chains_bwd<DV><<<2 * n, CHAIN_THREADS, smem, st>>>(m, n, (const bf*)q, (const bf*)k,
                                                     (const bf*)dout, S_in, dS_out, dS_in, ws);
  if ((e = cudaGetLastError())) return e;
  if ((e = tc_grad(m, DV, q, k, v, beta, dout, dq, dkk, dvv, dg, dbeta, ws, st))) return e;
  prof_mark(st, nullptr);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_fwd(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const float* S_in, void* o, float* S_out,
                   const TcWs& ws, const FwdSplit& sp, cudaStream_t st) {
  if (dv == 128) return fwd_t<128>(m, q, k, v, g, beta, S_in, o, S_out, ws, sp, st);
  return fwd_t<256>(m, q, k, v, g, beta, S_in, o, S_out, ws, sp, st);
}

cudaError_t tc_bwd(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const float* S_in, const void* dout,
                   const float* dS_out, void* dq, void* dkk, void* dvv, void* dg, void* dbeta,
                   float* dS_in, const TcWs& ws, bool run_pre, cudaStream_t st) {
  if (dv == 128)
    return bwd_t<128>(m, q, k, v, g, beta, S_in, dout, dS_out, dq, dkk, dvv, dg, dbeta, dS_in, ws,
                      run_pre, st);
  return bwd_t<256>(m, q, k, v, g, beta, S_in, dout, dS_out, dq, dkk, dvv, dg, dbeta, dS_in, ws,
                    run_pre, st);
}

}  // namespace gdn
