// Per-block gradient kernel of the bf16 tensor-core path: the reverse-mode
// derivative of one block's Pre / ST / Out (StateFlow review, Eq. 2; the
// backward rebuilds the trajectory Fwd consumed, Eq. 6) given H_b and V^new
// from the recompute chain (or from the forward that kept them) and
// dH_{b+1}, dV^new from the reverse chain (the same steps as the oracle's
// chunkwise module).
//
// Per block (t, s, r, c, u: tokens; Gamma_t = e^{gamma_t}; Mask_ts =
// e^{gamma_t - gamma_s} for s <= t):
//   OH = dO H_b^T-products, HW = dV^new H_b, Kt = V^new dH, OV = dO V^new^T,
//   WV = dV^new V^T (value-dimension reductions), Y = T^T dV^new,
//   P = OV * Mask, HK = HW K^T, dT = (WV - HK diag(Gamma)) diag(beta),
//   Z1 = T^T dT, dA = -strictly-lower(Z1 T^T), BE = diag(beta) (dA * Mask),
//   dq = diag(Gamma) OH + P K,
//   dk = diag(e^{gamma_C - gamma}) Kt + P^T Q - diag(beta Gamma) T^T HW + (BE + BE^T) K,
//   dv = diag(beta) Y, and the per-token sums that give dbeta and dgamma.
//
// Every product is a tcgen05 MMA (M = 128, N = 64) with its fp32 accumulator
// in tensor memory, issued by one thread from 128-byte-swizzled shared-memory
// tiles that TMA tensor copies fill straight from the workspace and the
// inputs. Products with 128 key rows fill the MMA's rows; a 64 x 64 product
// occupies the upper or lower 64 rows (the other half reads whatever tile
// follows its operand and is never used). Four epilogue warps share each
// 32-lane quarter of tensor memory and take 16 of the 64 columns each, so a
// thread owns a quarter row of every accumulator: key-row products give
// per-key rows, token-row products per-token rows whose sums stay in the
// thread (quarters combined through shared memory); the two sums over keys
// (q . OH, k . Kt) are butterflies over the warp's lanes. The kernel is persistent (one CTA
// per SM walks the block-heads) and every operand tile of the next
// block-head is loaded as soon as the current one has finished with its
// slot, so the copies run under the current block-head's products.
#include <cuda.h>

#include "gdn_internal.cuh"
#include "gdn_mma.cuh"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

constexpr uint32_t KB = 1024;
constexpr int NEPI = 512;        // epilogue threads: warps 0-15, four per TMEM lane quarter
constexpr int NTHR = NEPI + 32;  // + the control warp (TMA, MMA issue, TMEM allocation)
constexpr int CTL_WARP = NEPI / 32;

// Shared memory, byte offsets from a 1024-aligned base. Every tile is 64 bf16
// wide with 128-byte swizzled rows (8-row atoms of 1024 bytes).
namespace SL {
// one pass over 128 value columns
constexpr uint32_t HB = 0;            // H_b^T    [2 key halves][128 v][64 key]
constexpr uint32_t DH = 32 * KB;      // dH^T     [2 key halves][128 v][64 key]
constexpr uint32_t DO = 64 * KB;      // dO       [2 value chunks][64 t][64 v]
constexpr uint32_t VV = 80 * KB;      // V        [2 value chunks][64 s][64 v]
constexpr uint32_t VNT = 96 * KB;     // V^new^T  [128 v][64 t]
constexpr uint32_t DVNT = 112 * KB;   // dV^new^T [128 v][64 t]
constexpr uint32_t S_BYTES = 128 * KB;
// operands of the late products
constexpr uint32_t QQ = 128 * KB;     // Q [2 key halves][64 t][64 key]
constexpr uint32_t KK = 144 * KB;     // K [2 key halves][64 s][64 key]
constexpr uint32_t TT = 160 * KB;     // T [t][s]
constexpr uint32_t QKM = 168 * KB;    // Q K^T * Mask (Pre) [t][s]
constexpr uint32_t KKM = 176 * KB;    // K K^T * Mask, strictly lower (Pre) [r][c]
// tiles the epilogue writes
constexpr uint32_t DTT = 184 * KB;    // dT^T [s][t]; later Z1 [s][u]
constexpr uint32_t PT = 192 * KB;     // P [t][s]; later BE [r][c]
constexpr uint32_t HWT = 200 * KB;    // HW^T [128 key][64 t]
// per-block vectors, two buffers (block-heads alternate)
constexpr uint32_t DEC = 216 * KB;    // fp32 x 64 each: Gamma, e^{gamma_C - gamma}, gamma, beta
constexpr uint32_t VEC = DEC + 2 * KB;  // fp32 x 64 each: row, col, rho, db; then hd, Gamma_C
constexpr uint32_t VEC_STRIDE = 4 * 256 + 16;
// partial sums of one phase: [2 kinds][4 lane or column quarters][64] fp32, twice
constexpr uint32_t SCR = VEC + 2 * VEC_STRIDE;
constexpr uint32_t HDW = SCR + 4 * KB;  // [16]: <dH, H_b> per epilogue warp
constexpr uint32_t BAR = HDW + 64;
constexpr uint32_t BYTES = BAR + 128;
}  // namespace SL

// Tensor-memory columns (512 allocated). Late products reuse columns whose
// values the epilogue has consumed.
namespace TC {
constexpr uint32_t OH = 0, HW = 64, KT = 128, OV = 192, OVT = 256, WVT = 320, Y = 384;
constexpr uint32_t HKT = 192, DQ = 64, DK = 256, XG = 384, Z1 = 192, DA = 320, DAT = 192;
}  // namespace TC

constexpr uint32_t ID_KK = umma_idesc(128, 64, 0, 0);
constexpr uint32_t ID_KM = umma_idesc(128, 64, 0, 1);
constexpr uint32_t ID_MK = umma_idesc(128, 64, 1, 0);
constexpr uint32_t ID_MM = umma_idesc(128, 64, 1, 1);

// K-major operand (rows of the M / N dimension, 64 reduction elements each)
__device__ __forceinline__ uint64_t kdesc(uint32_t a) { return umma_desc(a, 16, 1024); }
// MN-major operand (rows of the reduction dimension; 64-wide M / N tiles lbo apart)
__device__ __forceinline__ uint64_t mdesc(uint32_t a, uint32_t lbo) { return umma_desc(a, lbo, 1024); }

// Byte offset of element (r, c) of a 64-wide swizzled tile.
__device__ __forceinline__ uint32_t sw64(int r, int c) {
  return (uint32_t)r * 128u + ((((uint32_t)c >> 3) ^ ((uint32_t)r & 7u)) << 4) + ((uint32_t)c & 7u) * 2u;
}
__device__ __forceinline__ float lds_bf(const unsigned char* p) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}
// 16 values -> bf16 into row r, columns [c0, c0 + 16) (c0 a multiple of 16) of a swizzled tile.
__device__ __forceinline__ void st_row16(unsigned char* tile, int r, int c0, const float* x) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint4 u;
    u.x = pack_bf16(x[8 * h], x[8 * h + 1]);
    u.y = pack_bf16(x[8 * h + 2], x[8 * h + 3]);
    u.z = pack_bf16(x[8 * h + 4], x[8 * h + 5]);
    u.w = pack_bf16(x[8 * h + 6], x[8 * h + 7]);
    *reinterpret_cast<uint4*>(tile + r * 128 + ((((c0 >> 3) + h) ^ (r & 7)) << 4)) = u;
  }
}
// Row r, columns [c0, c0 + 16) of a swizzled tile -> 16 floats.
__device__ __forceinline__ void ld_row16(const unsigned char* tile, int r, int c0, float* x) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 u = *reinterpret_cast<const uint4*>(tile + r * 128 + ((((c0 >> 3) + h) ^ (r & 7)) << 4));
    const float2 a = unpack_bf16(u.x), b = unpack_bf16(u.y), c = unpack_bf16(u.z), d = unpack_bf16(u.w);
    x[8 * h] = a.x;
    x[8 * h + 1] = a.y;
    x[8 * h + 2] = b.x;
    x[8 * h + 3] = b.y;
    x[8 * h + 4] = c.x;
    x[8 * h + 5] = c.y;
    x[8 * h + 6] = d.x;
    x[8 * h + 7] = d.y;
  }
}
// Column c, rows [r0, r0 + 16) of a swizzled tile -> 16 floats.
__device__ __forceinline__ void ld_col16(const unsigned char* tile, int r0, int c, float* x) {
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = lds_bf(tile + sw64(r0 + i, c));
}

// x[0..15] summed over the warp's 32 lanes by a butterfly that halves the
// vector at every step; lanes 2j and 2j + 1 return the sum of column j.
__device__ __forceinline__ float warp_colsum16(float* x) {
  const int l = threadIdx.x & 31;
#pragma unroll
  for (int o = 16, n = 8; o >= 2; o >>= 1, n >>= 1) {
    const bool hi = (l & o) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float send = hi ? x[i] : x[n + i];
      const float keep = hi ? x[n + i] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return x[0] + __shfl_xor_sync(0xffffffffu, x[0], 1);
}

template <class K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

struct GradMaps {
  CUtensorMap q, k, v, dout;                 // [B][T][H][d] views
  CUtensorMap hb, dh, vn, dvn, t;            // workspace views
};

template <int DV>
__global__ void __launch_bounds__(NTHR, 1)
    k_grad_tc(SeqMap m, TcWs ws, __nv_bfloat16* __restrict__ dq, __nv_bfloat16* __restrict__ dk,
              __nv_bfloat16* __restrict__ dvo, __nv_bfloat16* __restrict__ dg,
              __nv_bfloat16* __restrict__ dbeta, const __grid_constant__ GradMaps tm) {
  constexpr int NP = DV / 128;  // passes over 128 value columns
  static_assert(NP >= 1 && NP <= 2, "dv is 128 or 256");
  const int H = m.H, tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  const int total = m.nblk_cap * H;
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sb = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
  const uint32_t su = smem_u32(sb);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sb + SL::BAR);
  uint64_t* barS = bars + 0;    // one pass's H_b, dH, dO, V, V^new, dV^new
  uint64_t* barQ = bars + 1;    // Q
  uint64_t* barK = bars + 2;    // K
  uint64_t* barT = bars + 3;    // T
  uint64_t* barQM = bars + 4;   // Q K^T * Mask
  uint64_t* barKM = bars + 5;   // K K^T * Mask
  uint64_t* barD = bars + 6;    // decay vectors, one barrier per buffer (6, 7)
  uint64_t* barM = bars + 8;    // MMAs complete
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sb + SL::BAR + 80);
  volatile int* abort = reinterpret_cast<volatile int*>(sb + SL::BAR + 84);
  float* scr = reinterpret_cast<float*>(sb + SL::SCR);
  float* hdw = reinterpret_cast<float*>(sb + SL::HDW);
  const bool ctl = tid == NEPI;
  const int q4 = w & 3, cq = (w >> 2) & 3;  // TMEM lane quarter, 16-column quarter
  const int lane = 32 * q4 + l;             // TMEM lane = accumulator row of this thread
  const int c0 = 16 * cq;                   // this thread's accumulator columns [c0, c0 + 16)
  const bool epi = tid < NEPI;
  const bool upper = epi && q4 < 2, lower = epi && q4 >= 2;

  if (ctl) {
    for (int i = 0; i < 9; ++i) mbar_init(bars + i, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (w == CTL_WARP) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)c0;  // lane quarter, column quarter

  auto next_valid = [&](int it, BlockInfo& b) {
    while (it < total && !block_info(m, it / H, b)) it += gridDim.x;
    return it;
  };
  // ---- copies (control thread)
  auto tok_coord = [&](const BlockInfo& b, int& tc, int& sc) {
    tc = m.cu ? b.tok0 : b.lb * BT;  // token coordinate within the sequence
    sc = m.cu ? 0 : b.seq;
  };
  auto issue_s = [&](int it, const BlockInfo& b, int pass) {
    int tc, sc;
    tok_coord(b, tc, sc);
    const int h = it % H;
    mbar_arrive_expect_tx(barS, SL::S_BYTES);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      tma_load_3d(sb + SL::HB + c * 16 * KB, &tm.hb, 64 * c, 128 * pass, it, barS);
      tma_load_3d(sb + SL::DH + c * 16 * KB, &tm.dh, 64 * c, 128 * pass, it, barS);
      tma_load_4d(sb + SL::DO + c * 8 * KB, &tm.dout, 128 * pass + 64 * c, h, tc, sc, barS);
      tma_load_4d(sb + SL::VV + c * 8 * KB, &tm.v, 128 * pass + 64 * c, h, tc, sc, barS);
    }
    tma_load_3d(sb + SL::VNT, &tm.vn, 0, 128 * pass, it, barS);
    tma_load_3d(sb + SL::DVNT, &tm.dvn, 0, 128 * pass, it, barS);
  };
  auto issue_qk = [&](int it, const BlockInfo& b, uint32_t dst, const CUtensorMap* map, uint64_t* bar) {
    int tc, sc;
    tok_coord(b, tc, sc);
    mbar_arrive_expect_tx(bar, 16 * KB);
    tma_load_4d(sb + dst, map, 0, it % H, tc, sc, bar);
    tma_load_4d(sb + dst + 8 * KB, map, 64, it % H, tc, sc, bar);
  };
  auto issue_tile = [&](int it, uint32_t dst, const CUtensorMap* map, uint64_t* bar) {
    mbar_arrive_expect_tx(bar, 8 * KB);
    tma_load_3d(sb + dst, map, 0, 0, it, bar);
  };
  // Q K^T * Mask and K K^T * Mask: Pre writes them as swizzled tiles, copied as they are
  auto issue_msk = [&](int it, uint32_t dst, const __nv_bfloat16* src, uint64_t* bar) {
    mbar_arrive_expect_tx(bar, 8 * KB);
    bulk_g2s(sb + dst, src + (size_t)it * BT * TC_LD64, 8 * KB, bar);
  };
  auto issue_dec = [&](int it, int buf) {
    mbar_arrive_expect_tx(barD + buf, KB);
    bulk_g2s(sb + SL::DEC + buf * KB, ws.dec + (size_t)it * TC_DEC_ROWS * BT, KB, barD + buf);
  };
  auto mma = [&](uint32_t col, uint64_t a, uint64_t b, uint32_t id, bool acc) {
    umma_bf16(tmem + col, a, b, id, acc);
  };
  // token rows past a tail block's end read as zeros (the next sequence's rows
  // in a packed call, or the copy's zero fill past the tensor's end): rows
  // [len, 64) of the two 8 KB tiles at a and of the two at b
  auto zero_rows = [&](int len, uint32_t a, uint32_t b) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const int nr = BT - len;
    for (int idx = tid; idx < 4 * nr * 8; idx += NEPI) {
      const int tile = idx / (nr * 8), rem = idx - tile * nr * 8;
      const int r = len + (rem >> 3);
      const uint32_t base = (tile < 2 ? a : b) + (tile & 1) * 8 * KB;
      *reinterpret_cast<uint4*>(sb + base + r * 128 + (rem & 7) * 16) = z;
    }
  };
  // dgamma and dbeta of a finished block-head from its vectors (control warp)
  auto finish_vectors = [&](const float* v, int tok0, int len, int h) {
    const float *row = v, *col = v + BT, *rho = v + 2 * BT, *db = v + 3 * BT;
    const float hs = v[4 * BT], GC = v[4 * BT + 1];
    float rs = rho[l] + rho[l + 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
    // dgamma_r = row terms - column terms - rho_r; the gamma_C terms land on the last row
    float dgam0 = row[l] - col[l] - rho[l];
    float dgam1 = row[l + 32] - col[l + 32] - rho[l + 32];
    if (l == 31) dgam1 += rs + GC * hs;
    // reverse inclusive cumsum over 64 rows (fixed order)
    float a = dgam1, c = dgam0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float ya = __shfl_down_sync(0xffffffffu, a, off);
      const float yc = __shfl_down_sync(0xffffffffu, c, off);
      if (l + off < 32) {
        a += ya;
        c += yc;
      }
    }
    c += __shfl_sync(0xffffffffu, a, 0);
    if (l < len) {
      const size_t tok = (size_t)(tok0 + l) * H + h;
      dg[tok] = __float2bfloat16_rn(c);
      dbeta[tok] = __float2bfloat16_rn(db[l]);
    }
    if (l + 32 < len) {
      const size_t tok = (size_t)(tok0 + l + 32) * H + h;
      dg[tok] = __float2bfloat16_rn(a);
      dbeta[tok] = __float2bfloat16_rn(db[l + 32]);
    }
  };

  uint32_t dkp[8];  // the previous block-head's dk (this thread's key, 16 tokens), bf16 pairs
  // stores dkp for the block-head at (tok0_, len_, h_)
  auto store_dk = [&](int tok0_, int len_, int h_) {
    unsigned short* dst = reinterpret_cast<unsigned short*>(dk) + ((size_t)(tok0_ + c0) * H + h_) * 128 + lane;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (c0 + i < len_) dst[(size_t)i * H * 128] = (unsigned short)(dkp[i >> 1] >> (16 * (i & 1)));
  };
  uint32_t phS = 0, phQ = 0, phK = 0, phT = 0, phQM = 0, phKM = 0, phD = 0, phM = 0;  // phD: bit per buffer
  BlockInfo bi;
  int it = next_valid(blockIdx.x, bi);
  int buf = 0;
  bool prev = false;  // a finished block-head whose dgamma / dbeta are still to be written
  int ptok0 = 0, plen = 0, ph = 0;
  if (ctl && it < total) {
    issue_s(it, bi, 0);
    issue_qk(it, bi, SL::QQ, &tm.q, barQ);
    issue_qk(it, bi, SL::KK, &tm.k, barK);
    issue_tile(it, SL::TT, &tm.t, barT);
    issue_msk(it, SL::QKM, ws.QKM, barQM);
    issue_msk(it, SL::KKM, ws.KKM, barKM);
    issue_dec(it, 0);
  }
  while (it < total) {
    BlockInfo nbi;
    const int nit = next_valid(it + gridDim.x, nbi);
    const bool more = nit < total;
    const int h = it % H;
    const int len = bi.len, tok0 = bi.tok0;
    const float* dec = reinterpret_cast<const float*>(sb + SL::DEC + buf * KB);
    const float *sG = dec, *sDte = dec + BT, *sg = dec + 2 * BT, *sB = dec + 3 * BT;
    float* vec = reinterpret_cast<float*>(sb + SL::VEC + buf * SL::VEC_STRIDE);
    float* vrow = vec;           // per-token row terms of dgamma
    float* vcol = vec + BT;      // per-token column terms of dgamma
    float* vrho = vec + 2 * BT;  // e^{gamma_C - gamma_s} k_s . Kt_s
    float* vdb = vec + 3 * BT;   // dbeta
    if (tid < BT) {
      vrow[tid] = 0.f;
      vcol[tid] = 0.f;
      vdb[tid] = 0.f;
    }

    // ---- operands (most were prefetched while the previous block-head ran).
    // A wait that gives up sets the abort flag; the remaining steps then run on
    // whatever the tiles hold and the loop ends after this block-head.
    mbar_wait(barS, phS, abort);
    mbar_wait(barT, phT, abort);
    mbar_wait(barD + buf, (phD >> buf) & 1, abort);
    phS ^= 1;
    phT ^= 1;
    phD ^= 1u << buf;

    // ---- value-dimension products, one pass per 128 value columns
    float hd = 0.f;  // <dH, H_b> partial
#pragma unroll 1
    for (int p = 0; p < NP; ++p) {
      if (p > 0) {
        if (ctl) issue_s(it, bi, p);
        mbar_wait(barS, phS, abort);
        phS ^= 1;
      }
      if (len < BT && epi) zero_rows(len, SL::DO, SL::VV);
      fence_proxy_async_smem();
      __syncthreads();
      if (ctl) {
        tc_fence_after();
#pragma unroll 1
        for (int kk = 0; kk < 8; ++kk) {
          const bool acc = p > 0 || kk > 0;
          const uint32_t kb = (kk >> 2) * 8 * KB + 32 * (kk & 3);  // K-major step (value chunk, 16 columns)
          const uint32_t mr = 2048 * kk;                            // MN-major step (16 value rows)
          // OH^T [key][t] = H_b rows . dO
          mma(TC::OH, mdesc(su + SL::HB + mr, 16 * KB), kdesc(su + SL::DO + kb), ID_MK, acc);
          // HW^T [key][t] = H_b . dV^new^T
          mma(TC::HW, mdesc(su + SL::HB + mr, 16 * KB), mdesc(su + SL::DVNT + mr, 8 * KB), ID_MM, acc);
          // Kt^T [key][t] = dH . V^new^T
          mma(TC::KT, mdesc(su + SL::DH + mr, 16 * KB), mdesc(su + SL::VNT + mr, 8 * KB), ID_MM, acc);
          // OV [t][s] (rows 0-63)
          mma(TC::OV, kdesc(su + SL::DO + kb), mdesc(su + SL::VNT + mr, 8 * KB), ID_KM, acc);
          // OV^T [s][t] (rows 64-127)
          mma(TC::OVT, mdesc(su + SL::VNT + mr - 8 * KB, 8 * KB), kdesc(su + SL::DO + kb), ID_MK, acc);
          // WV^T [s][t] (rows 64-127)
          mma(TC::WVT, kdesc(su + SL::VV + kb - 8 * KB), mdesc(su + SL::DVNT + mr, 8 * KB), ID_KM, acc);
        }
        // Y^T [v][s] = dV^new^T T for this pass's 128 value rows
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma(TC::Y + 64 * p, kdesc(su + SL::DVNT + 32 * kk), mdesc(su + SL::TT + 2048 * kk, 8 * KB),
              ID_KM, kk > 0);
        umma_commit(barM);
      }
      if (epi) {
        if (prev && p == 0) store_dk(ptok0, plen, ph);  // the previous block-head's dk
        // <dH, H_b> over this pass: the two tiles share one layout
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t off = (uint32_t)(tid + NEPI * i) * 16u;
          const uint4 a = *reinterpret_cast<const uint4*>(sb + SL::HB + off);
          const uint4 b = *reinterpret_cast<const uint4*>(sb + SL::DH + off);
          const uint32_t* ap = &a.x;
          const uint32_t* bp = &b.x;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x = unpack_bf16(ap[e]), y = unpack_bf16(bp[e]);
            hd += x.x * y.x + x.y * y.y;
          }
        }
      } else if (prev && p == 0) {
        // the previous block-head's dgamma / dbeta (its vectors are final)
        finish_vectors(reinterpret_cast<const float*>(sb + SL::VEC + (buf ^ 1) * SL::VEC_STRIDE), ptok0,
                       plen, ph);
      }
      if (p == NP - 1) {
        // the operands of the later products, loaded under this block-head's first products
        mbar_wait(barQ, phQ, abort);
        mbar_wait(barK, phK, abort);
        mbar_wait(barQM, phQM, abort);
        mbar_wait(barKM, phKM, abort);
        phQ ^= 1;
        phK ^= 1;
        phQM ^= 1;
        phKM ^= 1;
        if (len < BT && epi) {
          zero_rows(len, SL::QQ, SL::KK);
          fence_proxy_async_smem();
        }
      }
      mbar_wait(barM, phM, abort);
      phM ^= 1;
      tc_fence_before();
      __syncthreads();  // the pass's tiles are free: MMAs complete, H_b / dH read
    }
    if (ctl && more) {
      issue_s(nit, nbi, 0);  // the next block-head's first pass
      issue_dec(nit, buf ^ 1);
    }
    tc_fence_after();

    // ---- E1: q . OH and k . Kt over keys; HW^T -> smem; dv; P and the sums of OV * QKM
    uint32_t dvp[NP][8];  // dv of this thread's value column(s), bf16 pairs
    if (epi) {
      const int key = lane;
      const uint32_t kt = (uint32_t)(key >> 6) * 8 * KB;
      const int kc = key & 63;
      float x[16], y[16], qv[16], kv[16];
      tmem_ld16(tl + TC::OH, x);
      tmem_ld16(tl + TC::KT, y);
      ld_col16(sb + SL::QQ + kt, c0, kc, qv);
      ld_col16(sb + SL::KK + kt, c0, kc, kv);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        x[i] *= qv[i];
        y[i] *= kv[i];
      }
      const float sq = warp_colsum16(x);
      const float sk = warp_colsum16(y);
      if (!(l & 1)) {
        scr[q4 * 64 + c0 + (l >> 1)] = sq;
        scr[256 + q4 * 64 + c0 + (l >> 1)] = sk;
      }
      tmem_ld16(tl + TC::HW, x);
      st_row16(sb + SL::HWT, key, c0, x);
      // dv = diag(beta) Y (Y^T rows are value columns), stored once the next products run
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        tmem_ld16(tl + TC::Y + 64 * p, x);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dvp[p][i] = pack_bf16(sB[c0 + 2 * i] * x[2 * i], sB[c0 + 2 * i + 1] * x[2 * i + 1]);
      }
      float acc = 0.f;
      if (upper) {
        // OV row t: P = OV * Mask; row sum of OV * QKM
        const int t = lane;
        const float gt = sg[t];
        tmem_ld16(tl + TC::OV, x);
        ld_row16(sb + SL::QKM, t, c0, y);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          acc += x[i] * y[i];
          // gamma is non-increasing, so the clamp only touches masked entries
          const float e = __expf(fminf(gt - sg[c0 + i], 0.f));
          x[i] = (c0 + i <= t ? x[i] : 0.f) * e;
        }
        st_row16(sb + SL::PT, t, c0, x);
        scr[512 + cq * 64 + t] = acc;
      } else {
        // OV^T row s: column sum of OV * QKM
        const int s = lane - 64;
        tmem_ld16(tl + TC::OVT, x);
        ld_col16(sb + SL::QKM, c0, s, y);
#pragma unroll
        for (int i = 0; i < 16; ++i) acc += x[i] * y[i];
        scr[768 + cq * 64 + s] = acc;
      }
      // <dH, H_b>: warp sum
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) hd += __shfl_xor_sync(0xffffffffu, hd, off);
      if (l == 0) hdw[w] = hd;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (ctl) {
      tc_fence_after();
      if (more) issue_msk(nit, SL::QKM, ws.QKM, barQM);  // Q K^T * Mask is read only above
      // HK^T [s][t] = K . HW^T (rows 64-127)
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma(TC::HKT, kdesc(su + SL::KK + (kk >> 2) * 8 * KB + 32 * (kk & 3) - 8 * KB),
            mdesc(su + SL::HWT + 2048 * kk, 8 * KB), ID_KM, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        // (P K)^T [key][t]
        mma(TC::DQ, mdesc(su + SL::KK + 2048 * kk, 8 * KB), kdesc(su + SL::PT + 32 * kk), ID_MK, kk > 0);
        // (P^T Q)^T [key][s]
        mma(TC::DK, mdesc(su + SL::QQ + 2048 * kk, 8 * KB), mdesc(su + SL::PT + 2048 * kk, 8 * KB), ID_MM,
            kk > 0);
        // (T^T HW)^T [key][s]
        mma(TC::XG, kdesc(su + SL::HWT + 32 * kk), mdesc(su + SL::TT + 2048 * kk, 8 * KB), ID_KM, kk > 0);
      }
      umma_commit(barM);
    }
    if (epi) {
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        unsigned short* dst =
            reinterpret_cast<unsigned short*>(dvo) + ((size_t)(tok0 + c0) * H + h) * DV + 128 * p + lane;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (c0 + i < len) dst[(size_t)i * H * DV] = (unsigned short)(dvp[p][i >> 1] >> (16 * (i & 1)));
      }
    }
    if (tid < BT) {
      const int t = tid;
      const float qo = scr[t] + scr[64 + t] + scr[128 + t] + scr[192 + t];
      const float ko = scr[256 + t] + scr[320 + t] + scr[384 + t] + scr[448 + t];
      vrow[t] += scr[512 + t] + scr[576 + t] + scr[640 + t] + scr[704 + t] + sG[t] * qo;
      vrho[t] = sDte[t] * ko;
      vcol[t] += scr[768 + t] + scr[832 + t] + scr[896 + t] + scr[960 + t];
      if (t == 0) {
        float hs = 0.f;
        for (int i = 0; i < NEPI / 32; ++i) hs += hdw[i];
        vec[4 * BT] = hs;
        vec[4 * BT + 1] = sG[BT - 1];
      }
    }
    if (epi) named_bar(1, NEPI);  // the partial sums are read: the scratch is free
    mbar_wait(barM, phM, abort);
    phM ^= 1;
    tc_fence_after();
    if (ctl && more) issue_qk(nit, nbi, SL::QQ, &tm.q, barQ);  // Q is free

    // ---- dq = diag(Gamma) OH + P K (key rows: one key column of 16 tokens per thread)
    //      E2 (rows s, lower): dT^T = diag(beta) (WV^T - diag(Gamma) HK^T); the T^T-weighted sums
    uint32_t dqp[8];  // dq of this thread's key, bf16 pairs; stored once Z1 runs
    if (epi) {
      float a[16], b[16];
      tmem_ld16(tl + TC::OH, a);
      tmem_ld16(tl + TC::DQ, b);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dqp[i] = pack_bf16(sG[c0 + 2 * i] * a[2 * i] + b[2 * i], sG[c0 + 2 * i + 1] * a[2 * i + 1] + b[2 * i + 1]);
    }
    if (lower) {
      const int s = lane - 64;
      const float bs = sB[s], Gs = sG[s];
      float wv[16], hk[16], tv[16];
      tmem_ld16(tl + TC::WVT, wv);
      tmem_ld16(tl + TC::HKT, hk);
      ld_col16(sb + SL::TT, c0, s, tv);
      float yv = 0.f, xk = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        yv += tv[i] * wv[i];  // sum_v Y[s][v] V[s][v]
        xk -= tv[i] * hk[i];  // k_s . x_s with x = -T^T HW
        wv[i] = bs * (wv[i] - Gs * hk[i]);
      }
      st_row16(sb + SL::DTT, s, c0, wv);
      scr[cq * 64 + s] = yv;
      scr[256 + cq * 64 + s] = xk;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (ctl) {
      tc_fence_after();
      // Z1 [s][u] = T^T dT (rows 0-63; the upper 64 rows read the dT^T tile)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma(TC::Z1, mdesc(su + SL::TT + 2048 * kk, SL::DTT - SL::TT), kdesc(su + SL::DTT + 32 * kk), ID_MK,
            kk > 0);
      umma_commit(barM);
    }
    if (epi) {
      unsigned short* dst = reinterpret_cast<unsigned short*>(dq) + ((size_t)(tok0 + c0) * H + h) * 128 + lane;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (c0 + i < len) dst[(size_t)i * H * 128] = (unsigned short)(dqp[i >> 1] >> (16 * (i & 1)));
    }
    if (tid >= BT && tid < 2 * BT) {
      const int s = tid - BT;
      const float yv = scr[s] + scr[64 + s] + scr[128 + s] + scr[192 + s];
      const float xk = scr[256 + s] + scr[320 + s] + scr[384 + s] + scr[448 + s];
      vdb[s] += yv + sG[s] * xk;
      vrow[s] += sB[s] * sG[s] * xk;
    }
    mbar_wait(barM, phM, abort);
    phM ^= 1;
    tc_fence_after();

    // ---- E3 (rows s, upper): Z1 -> smem
    if (upper) {
      float x[16];
      tmem_ld16(tl + TC::Z1, x);
      st_row16(sb + SL::DTT, lane, c0, x);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();  // (also: the E2 sums above are read, the scratch is free)
    if (ctl) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        // Z1 T^T [r][c] (rows 0-63) and T Z1^T [c][r] (rows 64-127)
        mma(TC::DA, kdesc(su + SL::DTT + 32 * kk), kdesc(su + SL::TT + 32 * kk), ID_KK, kk > 0);
        mma(TC::DAT, kdesc(su + SL::TT - 8 * KB + 32 * kk), kdesc(su + SL::DTT + 32 * kk), ID_KK, kk > 0);
      }
      umma_commit(barM);
    }
    mbar_wait(barM, phM, abort);
    phM ^= 1;
    tc_fence_after();
    if (ctl && more) issue_tile(nit, SL::TT, &tm.t, barT);  // T is free

    // ---- E4: dA = -strictly-lower(Z1 T^T); rows: dbeta, dgamma and BE; columns: dgamma
    if (upper) {
      const int r = lane;
      const float br = sB[r], gr = sg[r];
      float x[16], kk[16];
      tmem_ld16(tl + TC::DA, x);
      ld_row16(sb + SL::KKM, r, c0, kk);
      float sk = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float da = c0 + i < r ? -x[i] : 0.f;
        sk += da * kk[i];
        x[i] = br * da * __expf(fminf(gr - sg[c0 + i], 0.f));
      }
      st_row16(sb + SL::PT, r, c0, x);
      scr[cq * 64 + r] = sk;
    } else if (lower) {
      const int cc = lane - 64;
      float x[16], kv[16];
      tmem_ld16(tl + TC::DAT, x);
      ld_col16(sb + SL::KKM, c0, cc, kv);
      float cs = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) cs -= (c0 + i > cc ? sB[c0 + i] * x[i] : 0.f) * kv[i];
      scr[256 + cq * 64 + cc] = cs;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (ctl) {
      tc_fence_after();
      if (more) issue_msk(nit, SL::KKM, ws.KKM, barKM);  // K K^T * Mask is free
      // (BE + BE^T) K, transposed, onto (P^T Q)^T
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma(TC::DK, mdesc(su + SL::KK + 2048 * kk, 8 * KB), kdesc(su + SL::PT + 32 * kk), ID_MK, true);
        mma(TC::DK, mdesc(su + SL::KK + 2048 * kk, 8 * KB), mdesc(su + SL::PT + 2048 * kk, 8 * KB), ID_MM,
            true);
      }
      umma_commit(barM);
    }
    if (tid < BT) {
      const int r = tid;
      const float sk = scr[r] + scr[64 + r] + scr[128 + r] + scr[192 + r];
      vdb[r] += sk;
      vrow[r] += sB[r] * sk;
      vcol[r] += scr[256 + r] + scr[320 + r] + scr[384 + r] + scr[448 + r];
    }
    mbar_wait(barM, phM, abort);
    phM ^= 1;
    tc_fence_after();
    if (ctl && more) issue_qk(nit, nbi, SL::KK, &tm.k, barK);  // K is free

    // ---- dk = diag(e^{gamma_C - gamma}) Kt + (P^T Q + (BE + BE^T) K) - diag(beta Gamma) T^T HW,
    //      kept as bf16 pairs and stored while the next block-head's first products run
    if (epi) {
      float a[16], b[16], x[16];
      tmem_ld16(tl + TC::KT, a);
      tmem_ld16(tl + TC::DK, b);
      tmem_ld16(tl + TC::XG, x);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int s = c0 + i;
        a[i] = sDte[s] * a[i] + b[i] - sB[s] * sG[s] * x[i];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) dkp[i] = pack_bf16(a[2 * i], a[2 * i + 1]);
    }
    tc_fence_before();
    prev = true;
    ptok0 = tok0;
    plen = len;
    ph = h;
    buf ^= 1;
    if (__syncthreads_or(*abort != 0)) break;
    it = nit;
    bi = nbi;
  }
  if (epi && prev) store_dk(ptok0, plen, ph);
  if (w == CTL_WARP) {
    if (prev)
      finish_vectors(reinterpret_cast<const float*>(sb + SL::VEC + (buf ^ 1) * SL::VEC_STRIDE), ptok0, plen, ph);
    if (l == 0 && *abort) ws.status[0] = DEV_TIMEOUT;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (w == CTL_WARP) tmem_dealloc(tmem, 512);
}

template <int DV>
cudaError_t launch_grad(const SeqMap& m, const void* q, const void* k, const void* v,
                        const void* dout, void* dq, void* dkk, void* dvv, void* dg, void* dbeta,
                        const TcWs& ws, cudaStream_t st) {
  using bf = __nv_bfloat16;
  cudaError_t e;
  constexpr size_t smem = SL::BYTES + 1024;  // + alignment of the base
  if ((e = set_smem(k_grad_tc<DV>, smem))) return e;
  const long long items = (long long)m.nblk_cap * m.H;
  if (items <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) || (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)))
    return e;
  GradMaps tm;
  const long long nbh = items;
  if ((e = make_tok_map(&tm.q, q, 128, m)) || (e = make_tok_map(&tm.k, k, 128, m)) ||
      (e = make_tok_map(&tm.v, v, DV, m)) || (e = make_tok_map(&tm.dout, dout, DV, m)) ||
      (e = make_ws_map(&tm.hb, ws.HbT, 128, DV, 128, nbh, 128)) ||
      (e = make_ws_map(&tm.dh, ws.dHT, 128, DV, 128, nbh, 128)) ||
      (e = make_ws_map(&tm.vn, ws.VnT, BT, DV, BT, nbh, 128)) ||
      (e = make_ws_map(&tm.dvn, ws.dVnT, BT, DV, BT, nbh, 128)) ||
      (e = make_ws_map(&tm.t, ws.T, BT, BT, BT, nbh, BT)))
    return e;
  const int grid = (int)(items < sms ? items : sms);  // persistent: one CTA per SM
  prof_mark(st, "tc_grad");
  k_grad_tc<DV><<<grid, NTHR, smem, st>>>(m, ws, (bf*)dq, (bf*)dkk, (bf*)dvv, (bf*)dg, (bf*)dbeta, tm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_grad(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                    const void* beta, const void* dout, void* dq, void* dkk, void* dvv, void* dg,
                    void* dbeta, const TcWs& ws, cudaStream_t st) {
  (void)beta;
  if (dv == 128) return launch_grad<128>(m, q, k, v, dout, dq, dkk, dvv, dg, dbeta, ws, st);
  return launch_grad<256>(m, q, k, v, dout, dq, dkk, dvv, dg, dbeta, ws, st);
}

}  // namespace gdn
