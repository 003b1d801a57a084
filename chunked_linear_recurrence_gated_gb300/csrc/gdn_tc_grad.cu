// Per-block gradient kernel of the bf16 tensor-core path: the reverse-mode
// derivative of one block's Pre / ST / Out (StateFlow review, Eq. 2; the
// backward rebuilds the trajectory Fwd consumed, Eq. 6) given H_b and V^new
// from the recompute chain (or from the forward that kept them) and
// dH_{b+1}, dV^new from the reverse chain (the same steps as the oracle's
// chunkwise module).
#include "gdn_internal.cuh"
#include "gdn_mma.cuh"

namespace gdn {
namespace {

constexpr int LDK = TC_LDK;
constexpr int LD64 = TC_LD64;

// ------------------------------------------------------------------ per-block gradients
// 8 warps; warp (rw = w & 3, cw = w >> 2) owns rows [16 rw, 16 rw + 16) and
// key columns [64 cw, 64 cw + 64) of the 64 x 128 outputs, and columns
// [32 cw, 32 cw + 32) of the 64 x 64 ones. Value-dimension reductions stream
// over 64-column chunks.
constexpr int VC = 32;          // value columns per streamed chunk
constexpr int LDC = VC + 8;     // padded row of a [64][VC] chunk tile

struct GradChunk {
  __nv_bfloat16 dO[BT * LDC];
  __nv_bfloat16 V[BT * LDC];
  __nv_bfloat16 HbT[VC * LDK];
  __nv_bfloat16 dHT[VC * LDK];
  __nv_bfloat16 VnT[VC * LD64];
  __nv_bfloat16 dVnT[VC * LD64];
};
struct GradLate {                 // used only after the value-dimension loop
  __nv_bfloat16 HW[BT * LDK];     // dV^new H_b^T (= -dW)
  __nv_bfloat16 P[BT * LD64];     // (dO V^new^T) * Mask, later diag(beta) E
  __nv_bfloat16 X[BT * LD64];     // dT, later Z1 = T^T dT
};

struct GradBlk {                  // one block-head's operands (double-buffered across blocks)
  __nv_bfloat16 Q[BT * LDK];
  __nv_bfloat16 K[BT * LDK];
  __nv_bfloat16 T[BT * LD64];
  __nv_bfloat16 QKM[BT * LD64];   // Pre's Q K^T * Mask
  __nv_bfloat16 KKM[BT * LD64];   // Pre's K K^T * Mask
  float dec[TC_DEC_ROWS * BT];    // Gamma, e^{gamma_C - gamma}, gamma, beta
};

struct GradSmem {
  GradBlk blk[2];
  GradChunk ch[2];  // double-buffered value chunks; ch[1] doubles as GradLate after the loop
  float rowacc[2][BT];   // per column half
  float colacc[4][BT];   // per row quarter
  float dbeta[2][BT];
  float rho[2][BT];
  float red[8];
};
static_assert(sizeof(GradLate) <= sizeof(GradChunk), "late tiles overlay one chunk buffer");

__device__ __forceinline__ float quad_reduce(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}
// sum over the 8 row-groups (gq) of a warp
__device__ __forceinline__ float col_reduce(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  x += __shfl_xor_sync(0xffffffffu, x, 8);
  x += __shfl_xor_sync(0xffffffffu, x, 16);
  return x;
}

// Persistent: each CTA walks block-heads it = blockIdx.x, + gridDim.x, ...
// While one block-head's last value chunk and its late phases run, the next
// one's operands and first value chunk are already in flight.
template <int DV>
__global__ void __launch_bounds__(256, 1) k_grad_tc(SeqMap m, const __nv_bfloat16* __restrict__ q,
                                                    const __nv_bfloat16* __restrict__ k,
                                                    const __nv_bfloat16* __restrict__ v,
                                                    const __nv_bfloat16* __restrict__ dout,
                                                    __nv_bfloat16* __restrict__ dq,
                                                    __nv_bfloat16* __restrict__ dk,
                                                    __nv_bfloat16* __restrict__ dvo,
                                                    __nv_bfloat16* __restrict__ dg,
                                                    __nv_bfloat16* __restrict__ dbeta, TcWs ws) {
  constexpr int DK = 128;
  constexpr int NCH = DV / VC;
  static_assert(NCH % 2 == 0, "the last chunk must use buffer 1");
  const int H = m.H, tid = threadIdx.x;
  const int total = m.nblk_cap * H;
  extern __shared__ __align__(128) unsigned char smraw[];
  GradSmem& sm = *reinterpret_cast<GradSmem*>(smraw);
  GradLate& late = *reinterpret_cast<GradLate*>(&sm.ch[1]);
  const int w = tid >> 5, l = tid & 31, gq = l >> 2, tq = l & 3;
  const int rw = w & 3, cw = w >> 2;
  const int R0 = 16 * rw;

  auto next_valid = [&](int it, BlockInfo& b) {
    while (it < total && !block_info(m, it / H, b)) it += gridDim.x;
    return it;
  };
  // operands of block-head `it` into blk[buf] (no commit)
  auto load_blk = [&](int it, const BlockInfo& b, int buf) {
    GradBlk& B = sm.blk[buf];
    const int h = it % H;
    const size_t bh = (size_t)it;
    for (int idx = tid; idx < BT * 16; idx += 256) {
      const int r = idx >> 4, c = (idx & 15) * 8;
      const bool ok = r < b.len;
      const size_t off = ((size_t)(b.tok0 + (ok ? r : 0)) * H + h) * DK + c;
      cp16(&B.Q[r * LDK + c], q + off, ok);
      cp16(&B.K[r * LDK + c], k + off, ok);
    }
    for (int idx = tid; idx < BT * 8; idx += 256) {
      const int r = idx >> 3, c = (idx & 7) * 8;
      cp16(&B.T[r * LD64 + c], ws.T + bh * BT * BT + r * BT + c, true);
      cp16(&B.QKM[r * LD64 + c], ws.QKM + bh * BT * LD64 + r * LD64 + c, true);
      cp16(&B.KKM[r * LD64 + c], ws.KKM + bh * BT * LD64 + r * LD64 + c, true);
    }
    if (tid < TC_DEC_ROWS * BT / 4) cp16(&B.dec[4 * tid], ws.dec + bh * TC_DEC_ROWS * BT + 4 * tid, true);
  };
  // value chunk c of block-head `it` into ch[c & 1] (no commit)
  auto load_chunk = [&](int it, const BlockInfo& b, int c) {
    GradChunk& C = sm.ch[c & 1];
    const int h = it % H;
    const size_t bh = (size_t)it;
    const int v0 = c * VC;
    for (int idx = tid; idx < BT * (VC / 8); idx += 256) {
      const int r = idx / (VC / 8), cc = (idx % (VC / 8)) * 8;
      const bool ok = r < b.len;
      const size_t tok = (size_t)(b.tok0 + (ok ? r : 0)) * H + h;
      cp16(&C.dO[r * LDC + cc], dout + tok * DV + v0 + cc, ok);
      cp16(&C.V[r * LDC + cc], v + tok * DV + v0 + cc, ok);
    }
    for (int idx = tid; idx < VC * 8; idx += 256) {
      const int r = idx >> 3, cc = (idx & 7) * 8;
      cp16(&C.VnT[r * LD64 + cc], ws.VnT + bh * DV * BT + (size_t)(v0 + r) * BT + cc, true);
      cp16(&C.dVnT[r * LD64 + cc], ws.dVnT + bh * DV * BT + (size_t)(v0 + r) * BT + cc, true);
    }
    for (int idx = tid; idx < VC * 16; idx += 256) {
      const int r = idx >> 4, cc = (idx & 15) * 8;
      cp16(&C.HbT[r * LDK + cc], ws.HbT + bh * DV * DK + (size_t)(v0 + r) * DK + cc, true);
      cp16(&C.dHT[r * LDK + cc], ws.dHT + bh * DV * DK + (size_t)(v0 + r) * DK + cc, true);
    }
  };

  BlockInfo bi;
  int it = next_valid(blockIdx.x, bi);
  int buf = 0;
  if (it < total) {
    load_blk(it, bi, buf);
    load_chunk(it, bi, 0);
  }
  cp_commit();
  for (; it < total; buf ^= 1) {
  BlockInfo nbi;
  const int nit = next_valid(it + gridDim.x, nbi);
  const int h = it % H;
  const GradBlk& Bk = sm.blk[buf];
  const float* sG = Bk.dec;
  const float* sdte = Bk.dec + BT;
  const float* sg = Bk.dec + 2 * BT;
  const float* sb = Bk.dec + 3 * BT;
  for (int idx = tid; idx < 2 * BT; idx += 256) {
    (&sm.rowacc[0][0])[idx] = 0.f;
    (&sm.dbeta[0][0])[idx] = 0.f;
    (&sm.rho[0][0])[idx] = 0.f;
  }
  for (int idx = tid; idx < 4 * BT; idx += 256) (&sm.colacc[0][0])[idx] = 0.f;

  // ---- value-dimension reductions
  float aOH[8][4], aHW[8][4], aKt[8][4], aOV[4][4], aWV[4][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) aOH[j][e] = aHW[j][e] = aKt[j][e] = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) aOV[j][e] = aWV[j][e] = 0.f;
  float hd = 0.f;

  for (int c = 0; c < NCH; ++c) {
    if (c + 1 < NCH) {
      load_chunk(it, bi, c + 1);
    } else if (nit < total) {
      // the last chunk computes from ch[1]: ch[0] and the other operand buffer are free
      load_blk(nit, nbi, buf ^ 1);
      load_chunk(nit, nbi, 0);
    }
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    const GradChunk& C = sm.ch[c & 1];
#pragma unroll
    for (int kc = 0; kc < VC / 16; ++kc) {
      uint32_t aO[4], aW[4], aV[4], bH[4][4], bD[4][4], bN[2][4], bVv[2][4];
      lda_rm(aO, C.dO, LDC, R0, 16 * kc);       // dO   (token x value)
      lda_tr(aW, C.dVnT, LD64, R0, 16 * kc);    // dV^new
      lda_tr(aV, C.VnT, LD64, R0, 16 * kc);     // V^new
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        ldb_kn_x2n(bH[jj], C.HbT, LDK, 16 * kc, 64 * cw + 16 * jj);
        ldb_kn_x2n(bD[jj], C.dHT, LDK, 16 * kc, 64 * cw + 16 * jj);
      }
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        ldb_kn_x2n(bN[jj], C.VnT, LD64, 16 * kc, 32 * cw + 16 * jj);
        ldb_nk_x2n(bVv[jj], C.V, LDC, 32 * cw + 16 * jj, 16 * kc);
      }
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        mma16816(aOH[2 * jj], aO, bH[jj][0], bH[jj][1]);
        mma16816(aOH[2 * jj + 1], aO, bH[jj][2], bH[jj][3]);
        mma16816(aHW[2 * jj], aW, bH[jj][0], bH[jj][1]);
        mma16816(aHW[2 * jj + 1], aW, bH[jj][2], bH[jj][3]);
        mma16816(aKt[2 * jj], aV, bD[jj][0], bD[jj][1]);
        mma16816(aKt[2 * jj + 1], aV, bD[jj][2], bD[jj][3]);
      }
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        mma16816(aOV[2 * jj], aO, bN[jj][0], bN[jj][1]);
        mma16816(aOV[2 * jj + 1], aO, bN[jj][2], bN[jj][3]);
        mma16816(aWV[2 * jj], aW, bVv[jj][0], bVv[jj][1]);
        mma16816(aWV[2 * jj + 1], aW, bVv[jj][2], bVv[jj][3]);
      }
    }
    // <dH, H_b> partial
    for (int idx = tid; idx < VC * DK / 8; idx += 256) {
      const int r = idx >> 4, cc = (idx & 15) * 8;
      const uint4 a = *reinterpret_cast<const uint4*>(&C.dHT[r * LDK + cc]);
      const uint4 b = *reinterpret_cast<const uint4*>(&C.HbT[r * LDK + cc]);
      const uint32_t* ap = &a.x;
      const uint32_t* bp = &b.x;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = unpack_bf16(ap[e]), y = unpack_bf16(bp[e]);
        hd += x.x * y.x + x.y * y.y;
      }
    }
    // Y = T^T dV^new on this chunk (warp: rows R0.., value columns 16 cw..): dv = beta Y, dbeta += Y . V
    {
      float y[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) y[j][e] = 0.f;
      uint32_t at_[4][4], bY[4][4];
#pragma unroll
      for (int kc = 0; kc < 4; ++kc) {
        lda_tr(at_[kc], Bk.T, LD64, R0, 16 * kc);
        ldb_nk_x2n(bY[kc], C.dVnT, LD64, 16 * cw, 16 * kc);
      }
#pragma unroll
      for (int kc = 0; kc < 4; ++kc) {
        mma16816(y[0], at_[kc], bY[kc][0], bY[kc][1]);
        mma16816(y[1], at_[kc], bY[kc][2], bY[kc][3]);
      }
      float p0 = 0.f, p1 = 0.f;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int r = R0 + gq + 8 * hf, cc = 16 * cw + 8 * j + 2 * tq;
          const float2 vv = unpack_bf16(*reinterpret_cast<const uint32_t*>(&C.V[r * LDC + cc]));
          const float y0 = y[j][2 * hf], y1 = y[j][2 * hf + 1];
          if (r < bi.len)
            *reinterpret_cast<uint32_t*>(dvo + ((size_t)(bi.tok0 + r) * H + h) * DV + c * VC + cc) =
                pack_bf16(sb[r] * y0, sb[r] * y1);
          const float yv = y0 * vv.x + y1 * vv.y;
          if (hf == 0) p0 += yv; else p1 += yv;
        }
      p0 = quad_reduce(p0);
      p1 = quad_reduce(p1);
      if (tq == 0) {
        sm.dbeta[cw][R0 + gq] += p0;
        sm.dbeta[cw][R0 + gq + 8] += p1;
      }
    }
    __syncthreads();  // this buffer is refilled two chunks later
  }
  // block reduction of <dH, H_b>
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) hd += __shfl_xor_sync(0xffffffffu, hd, off);
  if (l == 0) sm.red[w] = hd;

  // this thread's two rows: per-row factors read once
  const int rr[2] = {R0 + gq, R0 + gq + 8};
  const float Gr[2] = {sG[rr[0]], sG[rr[1]]}, Dr[2] = {sdte[rr[0]], sdte[rr[1]]};
  const float Br[2] = {sb[rr[0]], sb[rr[1]]}, gr_[2] = {sg[rr[0]], sg[rr[1]]};
  // ---- dQ = Gamma dOH ; dgamma += Gamma q . dOH ; dK = dte dKt ; rho = dte k . dKt
  float aQ[8][4], aK[8][4];
  {
    float pq0 = 0.f, pq1 = 0.f, pk0 = 0.f, pk1 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = rr[hf], c = 64 * cw + 8 * j + 2 * tq;
        const float2 qv = unpack_bf16(*reinterpret_cast<const uint32_t*>(&Bk.Q[r * LDK + c]));
        const float2 kv = unpack_bf16(*reinterpret_cast<const uint32_t*>(&Bk.K[r * LDK + c]));
        const int e = 2 * hf;
        aQ[j][e] = Gr[hf] * aOH[j][e];
        aQ[j][e + 1] = Gr[hf] * aOH[j][e + 1];
        aK[j][e] = Dr[hf] * aKt[j][e];
        aK[j][e + 1] = Dr[hf] * aKt[j][e + 1];
        const float pq = qv.x * aOH[j][e] + qv.y * aOH[j][e + 1];
        const float pk = kv.x * aKt[j][e] + kv.y * aKt[j][e + 1];
        if (hf == 0) {
          pq0 += pq;
          pk0 += pk;
        } else {
          pq1 += pq;
          pk1 += pk;
        }
      }
    pq0 = quad_reduce(pq0);
    pq1 = quad_reduce(pq1);
    pk0 = quad_reduce(pk0);
    pk1 = quad_reduce(pk1);
    if (tq == 0) {
      sm.rowacc[cw][rr[0]] += Gr[0] * pq0;
      sm.rowacc[cw][rr[1]] += Gr[1] * pq1;
      sm.rho[cw][rr[0]] = Dr[0] * pk0;
      sm.rho[cw][rr[1]] = Dr[1] * pk1;
    }
    // HW -> smem (bf16)
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = R0 + gq + 8 * hf, c = 64 * cw + 8 * j + 2 * tq;
        *reinterpret_cast<uint32_t*>(&late.HW[r * LDK + c]) = pack_bf16(aHW[j][2 * hf], aHW[j][2 * hf + 1]);
      }
  }
  // ---- P = dOV * Mask -> smem ; R = P * (Q K^T) = dOV * QKM (Pre's masked Q K^T)
  //      -> row / column sums ; partial dT = beta_c dWV ; K K^T * Mask for the dA step
  float dT[4][4], kk[4][4];
  {
    const __nv_bfloat16* qkm = Bk.QKM;
    const __nv_bfloat16* kkm = Bk.KKM;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float cs0 = 0.f, cs1 = 0.f;
      const int c = 32 * cw + 8 * j + 2 * tq;
      const float2 gc = *reinterpret_cast<const float2*>(&sg[c]);
      const float2 bc = *reinterpret_cast<const float2*>(&sb[c]);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = rr[hf];
        const float2 qm = unpack_bf16(*reinterpret_cast<const uint32_t*>(qkm + r * LD64 + c));
        const float2 km = unpack_bf16(*reinterpret_cast<const uint32_t*>(kkm + r * LD64 + c));
        kk[j][2 * hf] = km.x;
        kk[j][2 * hf + 1] = km.y;
        const float m0 = (c <= r) ? __expf(gr_[hf] - gc.x) : 0.f;
        const float m1 = (c + 1 <= r) ? __expf(gr_[hf] - gc.y) : 0.f;
        const float R0v = aOV[j][2 * hf] * qm.x, R1v = aOV[j][2 * hf + 1] * qm.y;
        if (hf == 0) rs0 += R0v + R1v; else rs1 += R0v + R1v;
        cs0 += R0v;
        cs1 += R1v;
        aOV[j][2 * hf] *= m0;  // P in fp32
        aOV[j][2 * hf + 1] *= m1;
        *reinterpret_cast<uint32_t*>(&late.P[r * LD64 + c]) =
            pack_bf16(aOV[j][2 * hf], aOV[j][2 * hf + 1]);
        dT[j][2 * hf] = bc.x * aWV[j][2 * hf];
        dT[j][2 * hf + 1] = bc.y * aWV[j][2 * hf + 1];
      }
      cs0 = col_reduce(cs0);
      cs1 = col_reduce(cs1);
      if (gq == 0) {
        sm.colacc[rw][c] += cs0;
        sm.colacc[rw][c + 1] += cs1;
      }
    }
    rs0 = quad_reduce(rs0);
    rs1 = quad_reduce(rs1);
    if (tq == 0) {
      sm.rowacc[cw][R0 + gq] += rs0;
      sm.rowacc[cw][R0 + gq + 8] += rs1;
    }
  }
  __syncthreads();
  // ---- dT = beta_c dWV - beta_c Gamma_c (HW K^T) on this warp's 64 x 64 tile
  {
    float hk[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) hk[j][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < DK / 16; ++kc) {
      uint32_t ah_[4], b0[4], b1[4];
      lda_rm(ah_, late.HW, LDK, R0, 16 * kc);
      ldb_nk_x2n(b0, Bk.K, LDK, 32 * cw, 16 * kc);
      ldb_nk_x2n(b1, Bk.K, LDK, 32 * cw + 16, 16 * kc);
      mma16816(hk[0], ah_, b0[0], b0[1]);
      mma16816(hk[1], ah_, b0[2], b0[3]);
      mma16816(hk[2], ah_, b1[0], b1[1]);
      mma16816(hk[3], ah_, b1[2], b1[3]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = 32 * cw + 8 * j + 2 * tq;
      const float2 bc = *reinterpret_cast<const float2*>(&sb[c]);
      const float2 Gc = *reinterpret_cast<const float2*>(&sG[c]);
      const float f0 = bc.x * Gc.x, f1 = bc.y * Gc.y;
      dT[j][0] -= f0 * hk[j][0];
      dT[j][1] -= f1 * hk[j][1];
      dT[j][2] -= f0 * hk[j][2];
      dT[j][3] -= f1 * hk[j][3];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = R0 + gq + 8 * hf, c = 32 * cw + 8 * j + 2 * tq;
        *reinterpret_cast<uint32_t*>(&late.X[r * LD64 + c]) = pack_bf16(dT[j][2 * hf], dT[j][2 * hf + 1]);
      }
  }
  __syncthreads();
  // ---- dQ += P K ; dK += P^T Q ; Xg = -T^T HW -> dK, dbeta, dgamma ; Z1 = T^T dT
  {
    float xg[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) xg[j][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
      uint32_t ap[4], apt[4], att[4];
      lda_rm(ap, late.P, LD64, R0, 16 * kc);
      lda_tr(apt, late.P, LD64, R0, 16 * kc);
      lda_tr(att, Bk.T, LD64, R0, 16 * kc);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        uint32_t b[4];
        ldb_kn_x2n(b, Bk.K, LDK, 16 * kc, 64 * cw + 16 * jj);
        mma16816(aQ[2 * jj], ap, b[0], b[1]);
        mma16816(aQ[2 * jj + 1], ap, b[2], b[3]);
        ldb_kn_x2n(b, Bk.Q, LDK, 16 * kc, 64 * cw + 16 * jj);
        mma16816(aK[2 * jj], apt, b[0], b[1]);
        mma16816(aK[2 * jj + 1], apt, b[2], b[3]);
        ldb_kn_x2n(b, late.HW, LDK, 16 * kc, 64 * cw + 16 * jj);
        mma16816(xg[2 * jj], att, b[0], b[1]);
        mma16816(xg[2 * jj + 1], att, b[2], b[3]);
      }
    }
    float p0 = 0.f, p1 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = rr[hf], c = 64 * cw + 8 * j + 2 * tq;
        const float bg = Br[hf] * Gr[hf];
        const float2 kv = unpack_bf16(*reinterpret_cast<const uint32_t*>(&Bk.K[r * LDK + c]));
        const float x0 = -xg[j][2 * hf], x1 = -xg[j][2 * hf + 1];
        aK[j][2 * hf] += bg * x0;
        aK[j][2 * hf + 1] += bg * x1;
        const float kx = x0 * kv.x + x1 * kv.y;
        if (hf == 0) p0 += kx; else p1 += kx;
      }
    p0 = quad_reduce(p0);
    p1 = quad_reduce(p1);
    if (tq == 0) {
      sm.dbeta[cw][rr[0]] += Gr[0] * p0;
      sm.dbeta[cw][rr[1]] += Gr[1] * p1;
      sm.rowacc[cw][rr[0]] += Br[0] * Gr[0] * p0;
      sm.rowacc[cw][rr[1]] += Br[1] * Gr[1] * p1;
    }
  }
  float z1[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) z1[j][e] = 0.f;
#pragma unroll
  for (int kc = 0; kc < 4; ++kc) {
    uint32_t att[4], b[4];
    lda_tr(att, Bk.T, LD64, R0, 16 * kc);
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      ldb_kn_x2n(b, late.X, LD64, 16 * kc, 32 * cw + 16 * jj);
      mma16816(z1[2 * jj], att, b[0], b[1]);
      mma16816(z1[2 * jj + 1], att, b[2], b[3]);
    }
  }
  __syncthreads();  // everyone is done with P (as P) and X (as dT)
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int r = R0 + gq + 8 * hf, c = 32 * cw + 8 * j + 2 * tq;
      *reinterpret_cast<uint32_t*>(&late.X[r * LD64 + c]) = pack_bf16(z1[j][2 * hf], z1[j][2 * hf + 1]);
    }
  __syncthreads();
  // ---- dA = strictly-lower(-Z1 T^T); E = dA * Mask; BE = diag(beta) E
  {
    float da[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) da[j][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
      uint32_t a[4], b[4];
      lda_rm(a, late.X, LD64, R0, 16 * kc);
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        ldb_nk_x2n(b, Bk.T, LD64, 32 * cw + 16 * jj, 16 * kc);
        mma16816(da[2 * jj], a, b[0], b[1]);
        mma16816(da[2 * jj + 1], a, b[2], b[3]);
      }
    }
    float pb0 = 0.f, pb1 = 0.f, rg0 = 0.f, rg1 = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float cg0 = 0.f, cg1 = 0.f;
      const float2 gc = *reinterpret_cast<const float2*>(&sg[32 * cw + 8 * j + 2 * tq]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hf = e >> 1;
        const int r = rr[hf], c = 32 * cw + 8 * j + 2 * tq + (e & 1);
        const float dA = (c < r) ? -da[j][e] : 0.f;
        const float E = (c < r) ? dA * __expf(gr_[hf] - ((e & 1) ? gc.y : gc.x)) : 0.f;
        const float dAK = dA * kk[j][e];  // dA * K K^T * Mask = E * K K^T
        const float Gv = Br[hf] * dAK;
        if (e < 2) {
          pb0 += dAK;
          rg0 += Gv;
        } else {
          pb1 += dAK;
          rg1 += Gv;
        }
        if (e & 1) cg1 += Gv; else cg0 += Gv;
        da[j][e] = Br[hf] * E;
      }
      cg0 = col_reduce(cg0);
      cg1 = col_reduce(cg1);
      if (gq == 0) {
        const int c = 32 * cw + 8 * j + 2 * tq;
        sm.colacc[rw][c] += cg0;
        sm.colacc[rw][c + 1] += cg1;
      }
    }
    pb0 = quad_reduce(pb0);
    pb1 = quad_reduce(pb1);
    rg0 = quad_reduce(rg0);
    rg1 = quad_reduce(rg1);
    if (tq == 0) {
      const int r0 = R0 + gq, r1 = R0 + gq + 8;
      sm.dbeta[cw][r0] += pb0;
      sm.dbeta[cw][r1] += pb1;
      sm.rowacc[cw][r0] += rg0;
      sm.rowacc[cw][r1] += rg1;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = R0 + gq + 8 * hf, c = 32 * cw + 8 * j + 2 * tq;
        *reinterpret_cast<uint32_t*>(&late.P[r * LD64 + c]) = pack_bf16(da[j][2 * hf], da[j][2 * hf + 1]);
      }
  }
  __syncthreads();
  // ---- dK += (BE + BE^T) K
#pragma unroll
  for (int kc = 0; kc < 4; ++kc) {
    uint32_t a[4], at_[4];
    lda_rm(a, late.P, LD64, R0, 16 * kc);
    lda_tr(at_, late.P, LD64, R0, 16 * kc);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      uint32_t b[4];
      ldb_kn_x2n(b, Bk.K, LDK, 16 * kc, 64 * cw + 16 * jj);
      mma16816(aK[2 * jj], a, b[0], b[1]);
      mma16816(aK[2 * jj + 1], a, b[2], b[3]);
      mma16816(aK[2 * jj], at_, b[0], b[1]);
      mma16816(aK[2 * jj + 1], at_, b[2], b[3]);
    }
  }
  // ---- outputs
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int r = R0 + gq + 8 * hf, c = 64 * cw + 8 * j + 2 * tq;
      if (r < bi.len) {
        const size_t tok = (size_t)(bi.tok0 + r) * H + h;
        *reinterpret_cast<uint32_t*>(dq + tok * DK + c) = pack_bf16(aQ[j][2 * hf], aQ[j][2 * hf + 1]);
        *reinterpret_cast<uint32_t*>(dk + tok * DK + c) = pack_bf16(aK[j][2 * hf], aK[j][2 * hf + 1]);
      }
    }
  __syncthreads();
  if (tid < 32) {
    // dgamma_r = row terms - column terms - rho_r; the gamma_C terms land on the last row
    float hs = 0.f;
    for (int i = 0; i < 8; ++i) hs += sm.red[i];
    float rho = sm.rho[0][l] + sm.rho[1][l] + sm.rho[0][l + 32] + sm.rho[1][l + 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) rho += __shfl_xor_sync(0xffffffffu, rho, off);
    float dgam[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int r = l + 32 * hh;
      dgam[hh] = sm.rowacc[0][r] + sm.rowacc[1][r] - sm.colacc[0][r] - sm.colacc[1][r] -
                 sm.colacc[2][r] - sm.colacc[3][r] - sm.rho[0][r] - sm.rho[1][r];
    }
    if (l == 31) dgam[1] += rho + sG[BT - 1] * hs;
    // reverse inclusive cumsum over 64 rows (fixed order)
    float a = dgam[1], c = dgam[0];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float ya = __shfl_down_sync(0xffffffffu, a, off);
      const float yc = __shfl_down_sync(0xffffffffu, c, off);
      if (l + off < 32) {
        a += ya;
        c += yc;
      }
    }
    const float tot = __shfl_sync(0xffffffffu, a, 0);
    c += tot;
    const float db0 = sm.dbeta[0][l] + sm.dbeta[1][l];
    const float db1 = sm.dbeta[0][l + 32] + sm.dbeta[1][l + 32];
    if (l < bi.len) {
      const size_t tok = (size_t)(bi.tok0 + l) * H + h;
      dg[tok] = __float2bfloat16_rn(c);
      dbeta[tok] = __float2bfloat16_rn(db0);
    }
    if (l + 32 < bi.len) {
      const size_t tok = (size_t)(bi.tok0 + l + 32) * H + h;
      dg[tok] = __float2bfloat16_rn(a);
      dbeta[tok] = __float2bfloat16_rn(db1);
    }
  }
  __syncthreads();  // vectors, the late tiles and this operand buffer are reused next
  it = nit;
  bi = nbi;
  }
  cp_wait<0>();
}

template <class K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int DV>
cudaError_t launch_grad(const SeqMap& m, const void* q, const void* k, const void* v,
                        const void* beta, const void* dout, void* dq, void* dkk, void* dvv,
                        void* dg, void* dbeta, const TcWs& ws, cudaStream_t st) {
  using bf = __nv_bfloat16;
  cudaError_t e;
  if ((e = set_smem(k_grad_tc<DV>, sizeof(GradSmem)))) return e;
  const long long items = (long long)m.nblk_cap * m.H;
  if (items > 0) {
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) || (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)))
      return e;
    const int grid = (int)(items < sms ? items : sms);  // one resident CTA per SM
    prof_mark(st, "tc_grad");
    k_grad_tc<DV><<<grid, 256, sizeof(GradSmem), st>>>(
        m, (const bf*)q, (const bf*)k, (const bf*)v, (const bf*)dout, (bf*)dq, (bf*)dkk, (bf*)dvv,
        (bf*)dg, (bf*)dbeta, ws);
  }
  (void)beta;
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_grad(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                    const void* beta, const void* dout, void* dq, void* dkk, void* dvv, void* dg,
                    void* dbeta, const TcWs& ws, cudaStream_t st) {
  if (dv == 128) return launch_grad<128>(m, q, k, v, beta, dout, dq, dkk, dvv, dg, dbeta, ws, st);
  return launch_grad<256>(m, q, k, v, beta, dout, dq, dkk, dvv, dg, dbeta, ws, st);
}

}  // namespace gdn
