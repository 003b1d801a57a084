// fp32-arithmetic SIMT kernels of the chunkwise gated delta rule.
//
// These serve fp32 inputs (where the 1e-4 / 1e-3 tolerances rule out TF32 or
// bf16 tensor-core operands) and any shape the tensor-core kernels do not
// cover. All arithmetic is fp32 FFMA; inputs may be fp32 or bf16.
//
// Per 64-token block (local positions r, gamma_r = cumulative log-decay within
// the block, Gamma_r = exp(gamma_r), Mask_rj = exp(gamma_r - gamma_j), j <= r):
//   Pre : A = strictly-lower(diag(beta) K K^T * Mask), T = (I + A)^-1,
//         W = T diag(beta Gamma) K, U = T diag(beta) V
//   ST  : V^new = U - W H_b,  H_{b+1} = Gamma_C H_b + Kt^T V^new,
//         Kt_r = exp(gamma_C - gamma_r) k_r                (sequential)
//   Out : O = diag(Gamma) Q H_b + (Q K^T * Mask) V^new
// (StateFlow review: Pre / ST / Out decomposition with V^new, Eq. 2; the
// backward rebuilds the same trajectory from S_in, Eq. 6.) Only ratios
// exp(gamma_r - gamma_j) with j <= r and exp(gamma_C - gamma_r) are formed,
// so nothing overflows however strong the decay.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int NT = 256;  // threads per CTA for every SIMT kernel

template <typename TI>
__device__ void load_rows(float* s, int ld, const TI* __restrict__ X, int H, int h, int d,
                          int tok0, int len, int c0, int nc) {
  for (int idx = threadIdx.x; idx < BT * nc; idx += blockDim.x) {
    const int r = idx / nc, c = idx - r * nc;
    float x = 0.f;
    if (r < len) x = ldf(X + ((size_t)(tok0 + r) * H + h) * d + c0 + c);
    s[r * ld + c] = x;
  }
}

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

// ---------------------------------------------------------------- Pre
template <typename TI, int DK>
__global__ void __launch_bounds__(NT) k_pre(SeqMap m, int dv, const TI* __restrict__ k,
                                            const TI* __restrict__ v, const TI* __restrict__ g,
                                            const TI* __restrict__ beta, SimtWs ws) {
  BlockInfo bi;
  const int gb = blockIdx.x, h = blockIdx.y, H = m.H, tid = threadIdx.x;
  if (!block_info(m, gb, bi)) return;
  constexpr int LDK = DK + 1;
  extern __shared__ float sm[];
  float* sK = sm;               // BT x LDK
  float* sA = sK + BT * LDK;    // BT x 65
  float* sT = sA + BT * 65;     // BT x 65
  float* sV = sT + BT * 65;     // BT x 65
  float* sg = sV + BT * 65;     // BT
  float* sb = sg + BT;          // BT
  float* sbG = sb + BT;         // BT

  load_rows(sK, LDK, k, H, h, DK, bi.tok0, bi.len, 0, DK);
  if (tid < BT) {
    const bool ok = tid < bi.len;
    const size_t off = (size_t)(bi.tok0 + tid) * H + h;
    sg[tid] = ok ? ldf(g + off) : 0.f;
    sb[tid] = ok ? ldf(beta + off) : 0.f;
  }
  __syncthreads();
  if (tid == 0) {
    float a = 0.f;
    for (int r = 0; r < BT; ++r) {
      a += sg[r];
      sg[r] = a;
    }
  }
  __syncthreads();
  if (tid < BT) sbG[tid] = sb[tid] * expf(sg[tid]);
  for (int idx = tid; idx < BT * BT; idx += NT) {
    const int r = idx >> 6, j = idx & 63;
    float a = 0.f;
    if (j < r) {
      float d = 0.f;
#pragma unroll 8
      for (int i = 0; i < DK; ++i) d += sK[r * LDK + i] * sK[j * LDK + i];
      a = sb[r] * d * expf(sg[r] - sg[j]);
    }
    sA[r * 65 + j] = a;
  }
  __syncthreads();
  // T = (I + A)^-1 by forward substitution, one row per step.
  for (int r = 0; r < BT; ++r) {
    if (tid < BT) {
      const int c = tid;
      float t = (c == r) ? 1.f : 0.f;
      for (int j = c; j < r; ++j) t -= sA[r * 65 + j] * sT[j * 65 + c];
      sT[r * 65 + c] = t;
    }
    __syncthreads();
  }
  const size_t bh = (size_t)gb * H + h;
  if (ws.Tm)
    for (int idx = tid; idx < BT * BT; idx += NT) ws.Tm[bh * BT * BT + idx] = sT[(idx >> 6) * 65 + (idx & 63)];
  if (tid < BT) ws.gam[bh * BT + tid] = sg[tid];
  for (int idx = tid; idx < BT * DK; idx += NT) {
    const int r = idx / DK, i = idx - r * DK;
    float a = 0.f;
    for (int j = 0; j <= r; ++j) a += sT[r * 65 + j] * sbG[j] * sK[j * LDK + i];
    ws.W[bh * BT * DK + idx] = a;
  }
  for (int c0 = 0; c0 < dv; c0 += 64) {
    __syncthreads();
    load_rows(sV, 65, v, H, h, dv, bi.tok0, bi.len, c0, 64);
    __syncthreads();
    for (int idx = tid; idx < BT * 64; idx += NT) {
      const int r = idx >> 6, c = idx & 63;
      float a = 0.f;
      for (int j = 0; j <= r; ++j) a += sT[r * 65 + j] * sb[j] * sV[j * 65 + c];
      ws.U[(bh * BT + r) * dv + c0 + c] = a;
    }
  }
}

// ---------------------------------------------------------------- ST (forward chain)
constexpr int SBV = 16;  // value columns per chain CTA (the tile size BV of the review)

template <typename TI, int DK>
__global__ void __launch_bounds__(NT) k_st(SeqMap m, int dv, const TI* __restrict__ k,
                                           const float* S_in, float* S_out, SimtWs ws) {
  const int nvt = dv / SBV;
  const int tile = blockIdx.x % nvt;
  const int sh = blockIdx.x / nvt;
  const int H = m.H, h = sh % H, s = sh / H, tid = threadIdx.x;
  const SeqInfo si = seq_info(m, s);
  constexpr int LDK = DK + 1;
  extern __shared__ float sm[];
  float* sW = sm;               // BT x LDK
  float* sKt = sW + BT * LDK;   // BT x LDK
  float* sH = sKt + BT * LDK;   // DK x SBV
  float* sVn = sH + DK * SBV;   // BT x SBV
  float* sg = sVn + BT * SBV;   // BT
  const size_t sbase = ((size_t)s * H + h) * DK * dv + (size_t)tile * SBV;
  for (int idx = tid; idx < DK * SBV; idx += NT) {
    const int i = idx / SBV, c = idx - i * SBV;
    sH[idx] = S_in ? S_in[sbase + (size_t)i * dv + c] : 0.f;
  }
  for (int lb = 0; lb < si.nblk; ++lb) {
    const int gb = si.blk0 + lb, tok0 = si.tok0 + lb * BT, len = min(BT, si.len - lb * BT);
    const size_t bh = (size_t)gb * H + h;
    __syncthreads();
    for (int idx = tid; idx < DK * SBV; idx += NT) {
      const int i = idx / SBV, c = idx - i * SBV;
      ws.Hb[bh * DK * dv + (size_t)i * dv + tile * SBV + c] = sH[idx];
    }
    if (tid < BT) sg[tid] = ws.gam[bh * BT + tid];
    for (int idx = tid; idx < BT * DK; idx += NT) sW[(idx / DK) * LDK + idx % DK] = ws.W[bh * BT * DK + idx];
    load_rows(sKt, LDK, k, H, h, DK, tok0, len, 0, DK);
    __syncthreads();
    const float gC = sg[BT - 1];
    for (int idx = tid; idx < BT * DK; idx += NT) {
      const int r = idx / DK;
      sKt[r * LDK + idx % DK] *= expf(gC - sg[r]);
    }
    for (int idx = tid; idx < BT * SBV; idx += NT) {
      const int r = idx / SBV, c = idx - r * SBV;
      float x = 0.f;
#pragma unroll 8
      for (int i = 0; i < DK; ++i) x += sW[r * LDK + i] * sH[i * SBV + c];
      const float vn = ws.U[(bh * BT + r) * dv + tile * SBV + c] - x;
      sVn[idx] = vn;
      ws.Vn[(bh * BT + r) * dv + tile * SBV + c] = vn;
    }
    __syncthreads();
    const float GC = expf(gC);
    for (int idx = tid; idx < DK * SBV; idx += NT) {
      const int i = idx / SBV, c = idx - i * SBV;
      float a = 0.f;
#pragma unroll 8
      for (int r = 0; r < BT; ++r) a += sKt[r * LDK + i] * sVn[r * SBV + c];
      sH[idx] = GC * sH[idx] + a;
    }
  }
  __syncthreads();
  if (S_out)
    for (int idx = tid; idx < DK * SBV; idx += NT) {
      const int i = idx / SBV, c = idx - i * SBV;
      S_out[sbase + (size_t)i * dv + c] = sH[idx];
    }
}

// ---------------------------------------------------------------- Out
template <typename TI, int DK>
__global__ void __launch_bounds__(NT) k_out(SeqMap m, int dv, const TI* __restrict__ q,
                                            const TI* __restrict__ k, TI* __restrict__ o,
                                            SimtWs ws) {
  BlockInfo bi;
  const int gb = blockIdx.x, h = blockIdx.y, H = m.H, tid = threadIdx.x;
  if (!block_info(m, gb, bi)) return;
  constexpr int LDK = DK + 1;
  extern __shared__ float sm[];
  float* sQ = sm;               // BT x LDK
  float* sK = sQ + BT * LDK;    // BT x LDK
  float* sM = sK + BT * LDK;    // BT x 65  (Q K^T * Mask)
  float* sHt = sM + BT * 65;    // DK x 65  (Hb column tile)
  float* sVt = sHt + DK * 65;   // BT x 65  (V^new column tile)
  float* sg = sVt + BT * 65;    // BT
  const size_t bh = (size_t)gb * H + h;
  load_rows(sQ, LDK, q, H, h, DK, bi.tok0, bi.len, 0, DK);
  load_rows(sK, LDK, k, H, h, DK, bi.tok0, bi.len, 0, DK);
  if (tid < BT) sg[tid] = ws.gam[bh * BT + tid];
  __syncthreads();
  for (int idx = tid; idx < BT * BT; idx += NT) {
    const int r = idx >> 6, c = idx & 63;
    float a = 0.f;
    if (c <= r) {
#pragma unroll 8
      for (int i = 0; i < DK; ++i) a += sQ[r * LDK + i] * sK[c * LDK + i];
      a *= expf(sg[r] - sg[c]);
    }
    sM[r * 65 + c] = a;
  }
  for (int c0 = 0; c0 < dv; c0 += 64) {
    __syncthreads();
    for (int idx = tid; idx < DK * 64; idx += NT) {
      const int i = idx >> 6, c = idx & 63;
      sHt[i * 65 + c] = ws.Hb[bh * DK * dv + (size_t)i * dv + c0 + c];
    }
    for (int idx = tid; idx < BT * 64; idx += NT) {
      const int r = idx >> 6, c = idx & 63;
      sVt[r * 65 + c] = ws.Vn[(bh * BT + r) * dv + c0 + c];
    }
    __syncthreads();
    for (int idx = tid; idx < BT * 64; idx += NT) {
      const int r = idx >> 6, c = idx & 63;
      if (r >= bi.len) continue;
      float a1 = 0.f, a2 = 0.f;
#pragma unroll 8
      for (int i = 0; i < DK; ++i) a1 += sQ[r * LDK + i] * sHt[i * 65 + c];
      for (int j = 0; j <= r; ++j) a2 += sM[r * 65 + j] * sVt[j * 65 + c];
      stf(o + ((size_t)(bi.tok0 + r) * H + h) * dv + c0 + c, expf(sg[r]) * a1 + a2);
    }
  }
}

// ---------------------------------------------------------------- ST backward (reverse chain)
// dV^new_b = (Q K^T * Mask)^T dO_b + Kt dH_{b+1}
// dH_b     = Gamma_C dH_{b+1} + (diag(Gamma) Q)^T dO_b - W^T dV^new_b
template <typename TI, int DK>
__global__ void __launch_bounds__(NT) k_st_bwd(SeqMap m, int dv, const TI* __restrict__ q,
                                               const TI* __restrict__ k,
                                               const TI* __restrict__ dout, const float* dS_out,
                                               float* dS_in, SimtWs ws) {
  const int nvt = dv / SBV;
  const int tile = blockIdx.x % nvt;
  const int sh = blockIdx.x / nvt;
  const int H = m.H, h = sh % H, s = sh / H, tid = threadIdx.x;
  const SeqInfo si = seq_info(m, s);
  constexpr int LDK = DK + 1;
  extern __shared__ float sm[];
  float* sQ = sm;               // BT x LDK (scaled by Gamma)
  float* sKt = sQ + BT * LDK;   // BT x LDK
  float* sW = sKt + BT * LDK;   // BT x LDK
  float* sM = sW + BT * LDK;    // BT x 65
  float* sdH = sM + BT * 65;    // DK x SBV
  float* sdO = sdH + DK * SBV;  // BT x SBV
  float* sdV = sdO + BT * SBV;  // BT x SBV
  float* sg = sdV + BT * SBV;   // BT
  const size_t sbase = ((size_t)s * H + h) * DK * dv + (size_t)tile * SBV;
  for (int idx = tid; idx < DK * SBV; idx += NT) {
    const int i = idx / SBV, c = idx - i * SBV;
    sdH[idx] = dS_out ? dS_out[sbase + (size_t)i * dv + c] : 0.f;
  }
  for (int lb = si.nblk - 1; lb >= 0; --lb) {
    const int gb = si.blk0 + lb, tok0 = si.tok0 + lb * BT, len = min(BT, si.len - lb * BT);
    const size_t bh = (size_t)gb * H + h;
    __syncthreads();
    for (int idx = tid; idx < DK * SBV; idx += NT) {
      const int i = idx / SBV, c = idx - i * SBV;
      ws.dH[bh * DK * dv + (size_t)i * dv + tile * SBV + c] = sdH[idx];
    }
    load_rows(sQ, LDK, q, H, h, DK, tok0, len, 0, DK);
    load_rows(sKt, LDK, k, H, h, DK, tok0, len, 0, DK);
    load_rows(sdO, SBV, dout, H, h, dv, tok0, len, tile * SBV, SBV);
    for (int idx = tid; idx < BT * DK; idx += NT) sW[(idx / DK) * LDK + idx % DK] = ws.W[bh * BT * DK + idx];
    if (tid < BT) sg[tid] = ws.gam[bh * BT + tid];
    __syncthreads();
    for (int idx = tid; idx < BT * BT; idx += NT) {
      const int r = idx >> 6, c = idx & 63;
      float a = 0.f;
      if (c <= r) {
#pragma unroll 8
        for (int i = 0; i < DK; ++i) a += sQ[r * LDK + i] * sKt[c * LDK + i];
        a *= expf(sg[r] - sg[c]);
      }
      sM[r * 65 + c] = a;
    }
    __syncthreads();
    const float gC = sg[BT - 1];
    for (int idx = tid; idx < BT * DK; idx += NT) {
      const int r = idx / DK, i = idx - r * DK;
      sQ[r * LDK + i] *= expf(sg[r]);
      sKt[r * LDK + i] *= expf(gC - sg[r]);
    }
    __syncthreads();
    for (int idx = tid; idx < BT * SBV; idx += NT) {
      const int r = idx / SBV, c = idx - r * SBV;
      float a = 0.f;
      for (int rr = r; rr < BT; ++rr) a += sM[rr * 65 + r] * sdO[rr * SBV + c];
#pragma unroll 8
      for (int i = 0; i < DK; ++i) a += sKt[r * LDK + i] * sdH[i * SBV + c];
      sdV[idx] = a;
      ws.dVn[(bh * BT + r) * dv + tile * SBV + c] = a;
    }
    __syncthreads();
    const float GC = expf(gC);
    for (int idx = tid; idx < DK * SBV; idx += NT) {
      const int i = idx / SBV, c = idx - i * SBV;
      float a = 0.f;
#pragma unroll 8
      for (int r = 0; r < BT; ++r) a += sQ[r * LDK + i] * sdO[r * SBV + c] - sW[r * LDK + i] * sdV[r * SBV + c];
      sdH[idx] = GC * sdH[idx] + a;
    }
  }
  __syncthreads();
  if (dS_in)
    for (int idx = tid; idx < DK * SBV; idx += NT) {
      const int i = idx / SBV, c = idx - i * SBV;
      dS_in[sbase + (size_t)i * dv + c] = sdH[idx];
    }
}

// ---------------------------------------------------------------- per-block gradients
// Reverse-mode derivative of one block's Pre / ST / Out given H_b, dH_{b+1},
// V^new and dV^new (see the derivation in the oracle's chunkwise module).
constexpr int GT = 16;  // column tile of the staged passes

template <typename TI, int DK>
__global__ void __launch_bounds__(NT) k_grad(SeqMap m, int dv, const TI* __restrict__ q,
                                             const TI* __restrict__ k, const TI* __restrict__ v,
                                             const TI* __restrict__ beta,
                                             const TI* __restrict__ dout, TI* __restrict__ dq,
                                             TI* __restrict__ dk, TI* __restrict__ dvo,
                                             TI* __restrict__ dg, TI* __restrict__ dbeta,
                                             SimtWs ws) {
  BlockInfo bi;
  const int gb = blockIdx.x, h = blockIdx.y, H = m.H, tid = threadIdx.x;
  if (!block_info(m, gb, bi)) return;
  constexpr int LDK = DK + 1;
  constexpr int NI = DK / 4;
  constexpr int LDT = GT + 1;
  extern __shared__ float sm[];
  float* sQ = sm;                  // BT x LDK
  float* sK = sQ + BT * LDK;       // BT x LDK
  float* sHW = sK + BT * LDK;      // BT x LDK   HW = dV^new Hb^T = -dW
  float* sM = sHW + BT * LDK;      // BT x 65    decay mask (j <= r)
  float* sT = sM + BT * 65;        // BT x 65
  float* sP = sT + BT * 65;        // BT x 65
  float* sX = sP + BT * 65;        // BT x 65
  float* sY = sX + BT * 65;        // BT x 65
  float* sA1 = sY + BT * 65;       // DK x LDT   staged Hb / dH column tile
  float* sA2 = sA1 + DK * LDT;     // DK x LDT   staged dH column tile
  float* sB1 = sA2 + DK * LDT;     // BT x LDT
  float* sB2 = sB1 + BT * LDT;     // BT x LDT
  float* sB3 = sB2 + BT * LDT;     // BT x LDT
  float* sg = sB3 + BT * LDT;      // BT
  float* sG = sg + BT;             // BT  Gamma
  float* sb = sG + BT;             // BT  beta
  float* sdte = sb + BT;           // BT  exp(gamma_C - gamma_r)
  float* sdgam = sdte + BT;        // BT  d gamma accumulator
  float* sdb = sdgam + BT;         // BT  d beta accumulator
  float* srho = sdb + BT;          // BT
  float* sred = srho + BT;         // NT / 32 partial sums

  const size_t bh = (size_t)gb * H + h;
  const int r = tid >> 2, q4 = tid & 3;
  const float* Hb = ws.Hb + bh * DK * dv;
  const float* dHn = ws.dH + bh * DK * dv;
  const float* Vn = ws.Vn + bh * BT * dv;
  const float* dVn = ws.dVn + bh * BT * dv;

  load_rows(sQ, LDK, q, H, h, DK, bi.tok0, bi.len, 0, DK);
  load_rows(sK, LDK, k, H, h, DK, bi.tok0, bi.len, 0, DK);
  if (tid < BT) {
    sg[tid] = ws.gam[bh * BT + tid];
    sb[tid] = tid < bi.len ? ldf(beta + (size_t)(bi.tok0 + tid) * H + h) : 0.f;
    sdgam[tid] = 0.f;
    sdb[tid] = 0.f;
  }
  for (int idx = tid; idx < BT * BT; idx += NT) sT[(idx >> 6) * 65 + (idx & 63)] = ws.Tm[bh * BT * BT + idx];
  __syncthreads();
  if (tid < BT) {
    sG[tid] = expf(sg[tid]);
    sdte[tid] = expf(sg[BT - 1] - sg[tid]);
  }
  for (int idx = tid; idx < BT * BT; idx += NT) {
    const int rr = idx >> 6, c = idx & 63;
    sM[rr * 65 + c] = c <= rr ? expf(sg[rr] - sg[c]) : 0.f;
  }

  float aQ[NI], aK[NI];
  // Pass A: dOH = dO Hb^T, HW = dV^new Hb^T, <dH, Hb>
  float hd = 0.f;
  {
    float aOH[NI], aHW[NI];
#pragma unroll
    for (int mi = 0; mi < NI; ++mi) aOH[mi] = aHW[mi] = 0.f;
    for (int j0 = 0; j0 < dv; j0 += GT) {
      __syncthreads();
      for (int idx = tid; idx < DK * GT; idx += NT) {
        const int i = idx / GT, jj = idx - i * GT;
        sA1[i * LDT + jj] = Hb[(size_t)i * dv + j0 + jj];
        sA2[i * LDT + jj] = dHn[(size_t)i * dv + j0 + jj];
      }
      load_rows(sB1, LDT, dout, H, h, dv, bi.tok0, bi.len, j0, GT);
      for (int idx = tid; idx < BT * GT; idx += NT) {
        const int rr = idx / GT, jj = idx - rr * GT;
        sB2[rr * LDT + jj] = dVn[(size_t)rr * dv + j0 + jj];
      }
      __syncthreads();
      for (int jj = 0; jj < GT; ++jj) {
        const float o_ = sB1[r * LDT + jj], w_ = sB2[r * LDT + jj];
#pragma unroll
        for (int mi = 0; mi < NI; ++mi) {
          const float hb = sA1[(q4 + 4 * mi) * LDT + jj];
          aOH[mi] += o_ * hb;
          aHW[mi] += w_ * hb;
        }
      }
      for (int idx = tid; idx < DK * GT; idx += NT) {
        const int i = idx / GT, jj = idx - i * GT;
        hd += sA1[i * LDT + jj] * sA2[i * LDT + jj];
      }
    }
    float part = 0.f;
#pragma unroll
    for (int mi = 0; mi < NI; ++mi) {
      const int i = q4 + 4 * mi;
      aQ[mi] = sG[r] * aOH[mi];
      part += sQ[r * LDK + i] * aOH[mi];
      sHW[r * LDK + i] = aHW[mi];
    }
    part = quad_sum(part);
    if (q4 == 0) sdgam[r] += sG[r] * part;
  }
  // block reduction of <dH, Hb> (fixed order)
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) hd += __shfl_xor_sync(0xffffffffu, hd, off);
  if ((tid & 31) == 0) sred[tid >> 5] = hd;

  // Pass B: dKt = V^new dH^T, dOV = dO V^new^T, dWV = dV^new V^T
  {
    float aKt[NI], aOV[16], aWV[16];
#pragma unroll
    for (int mi = 0; mi < NI; ++mi) aKt[mi] = 0.f;
#pragma unroll
    for (int mc = 0; mc < 16; ++mc) aOV[mc] = aWV[mc] = 0.f;
    for (int j0 = 0; j0 < dv; j0 += GT) {
      __syncthreads();
      for (int idx = tid; idx < DK * GT; idx += NT) {
        const int i = idx / GT, jj = idx - i * GT;
        sA2[i * LDT + jj] = dHn[(size_t)i * dv + j0 + jj];
      }
      for (int idx = tid; idx < BT * GT; idx += NT) {
        const int rr = idx / GT, jj = idx - rr * GT;
        sA1[rr * LDT + jj] = Vn[(size_t)rr * dv + j0 + jj];
        sB2[rr * LDT + jj] = dVn[(size_t)rr * dv + j0 + jj];
      }
      load_rows(sB1, LDT, dout, H, h, dv, bi.tok0, bi.len, j0, GT);
      load_rows(sB3, LDT, v, H, h, dv, bi.tok0, bi.len, j0, GT);
      __syncthreads();
      for (int jj = 0; jj < GT; ++jj) {
        const float vn = sA1[r * LDT + jj], o_ = sB1[r * LDT + jj], w_ = sB2[r * LDT + jj];
#pragma unroll
        for (int mi = 0; mi < NI; ++mi) aKt[mi] += vn * sA2[(q4 + 4 * mi) * LDT + jj];
#pragma unroll
        for (int mc = 0; mc < 16; ++mc) {
          const int c = q4 + 4 * mc;
          aOV[mc] += o_ * sA1[c * LDT + jj];
          aWV[mc] += w_ * sB3[c * LDT + jj];
        }
      }
    }
    float part = 0.f;
#pragma unroll
    for (int mi = 0; mi < NI; ++mi) {
      const int i = q4 + 4 * mi;
      aK[mi] = sdte[r] * aKt[mi];
      part += sK[r * LDK + i] * aKt[mi];
    }
    part = quad_sum(part);
    if (q4 == 0) srho[r] = sdte[r] * part;
#pragma unroll
    for (int mc = 0; mc < 16; ++mc) {
      const int c = q4 + 4 * mc;
      sP[r * 65 + c] = aOV[mc] * sM[r * 65 + c];
      sX[r * 65 + c] = sb[c] * aWV[mc];
    }
  }
  __syncthreads();
  if (q4 == 0) sdgam[r] -= srho[r];
  // dT = dW (beta Gamma K)^T + dV^new (beta V)^T  (sX holds the second term);
  // R = P * (Q K^T) into sY; KK = K K^T kept in registers.
  float kk[16];
#pragma unroll
  for (int mc = 0; mc < 16; ++mc) {
    const int c = q4 + 4 * mc;
    float a = 0.f, qk = 0.f, kk_ = 0.f;
#pragma unroll 8
    for (int i = 0; i < DK; ++i) {
      const float kc = sK[c * LDK + i];
      a += sHW[r * LDK + i] * kc;
      qk += sQ[r * LDK + i] * kc;
      kk_ += sK[r * LDK + i] * kc;
    }
    sX[r * 65 + c] -= sb[c] * sG[c] * a;
    sY[r * 65 + c] = sP[r * 65 + c] * qk;
    kk[mc] = kk_;
  }
  __syncthreads();
  if (tid < BT) {
    float rs = 0.f, cs = 0.f;
    for (int c = 0; c < BT; ++c) {
      rs += sY[tid * 65 + c];
      cs += sY[c * 65 + tid];
    }
    sdgam[tid] += rs - cs;
  }
  // dQ += P K, dK += P^T Q; X = T^T dW = -T^T HW
  {
    float part = 0.f;
#pragma unroll
    for (int mi = 0; mi < NI; ++mi) {
      const int i = q4 + 4 * mi;
      float a = 0.f, b = 0.f, x = 0.f;
      for (int c = 0; c < BT; ++c) {
        a += sP[r * 65 + c] * sK[c * LDK + i];
        b += sP[c * 65 + r] * sQ[c * LDK + i];
        x -= sT[c * 65 + r] * sHW[c * LDK + i];
      }
      aQ[mi] += a;
      aK[mi] += b + sb[r] * sG[r] * x;
      part += x * sK[r * LDK + i];
    }
    part = quad_sum(part);
    __syncthreads();
    if (q4 == 0) {
      sdb[r] += sG[r] * part;
      sdgam[r] += sb[r] * sG[r] * part;
    }
  }
  // Z1 = T^T dT
  float z[16];
#pragma unroll
  for (int mc = 0; mc < 16; ++mc) {
    const int c = q4 + 4 * mc;
    float a = 0.f;
    for (int mm = 0; mm < BT; ++mm) a += sT[mm * 65 + r] * sX[mm * 65 + c];
    z[mc] = a;
  }
  __syncthreads();
#pragma unroll
  for (int mc = 0; mc < 16; ++mc) sY[r * 65 + q4 + 4 * mc] = z[mc];
  __syncthreads();
  // dA = strictly-lower(-Z1 T^T); E = dA * Mask; BE = diag(beta) E; G = dA * A
  {
    float pb = 0.f, rowG = 0.f;
#pragma unroll
    for (int mc = 0; mc < 16; ++mc) {
      const int c = q4 + 4 * mc;
      float dA = 0.f;
      if (c < r)
        for (int mm = 0; mm < BT; ++mm) dA -= sY[r * 65 + mm] * sT[c * 65 + mm];
      const float E = dA * sM[r * 65 + c];
      const float G = sb[r] * E * kk[mc];
      pb += E * kk[mc];
      rowG += G;
      z[mc] = G;
      sP[r * 65 + c] = sb[r] * E;  // P is no longer needed
    }
    pb = quad_sum(pb);
    rowG = quad_sum(rowG);
    __syncthreads();
#pragma unroll
    for (int mc = 0; mc < 16; ++mc) sX[r * 65 + q4 + 4 * mc] = z[mc];
    if (q4 == 0) {
      sdb[r] += pb;
      sdgam[r] += rowG;
    }
  }
  __syncthreads();
  if (tid < BT) {
    float cs = 0.f;
    for (int rr = 0; rr < BT; ++rr) cs += sX[rr * 65 + tid];
    sdgam[tid] -= cs;
  }
#pragma unroll
  for (int mi = 0; mi < NI; ++mi) {
    const int i = q4 + 4 * mi;
    float a = 0.f;
    for (int c = 0; c < BT; ++c) a += (sP[r * 65 + c] + sP[c * 65 + r]) * sK[c * LDK + i];
    aK[mi] += a;
  }
  // Y = T^T dV^new: dv = beta Y, dbeta += Y . V
  {
    float part = 0.f;
    for (int j0 = 0; j0 < dv; j0 += GT) {
      __syncthreads();
      for (int idx = tid; idx < BT * GT; idx += NT) {
        const int rr = idx / GT, jj = idx - rr * GT;
        sB2[rr * LDT + jj] = dVn[(size_t)rr * dv + j0 + jj];
      }
      load_rows(sB3, LDT, v, H, h, dv, bi.tok0, bi.len, j0, GT);
      __syncthreads();
#pragma unroll
      for (int mj = 0; mj < GT / 4; ++mj) {
        const int jj = q4 + 4 * mj;
        float y = 0.f;
        for (int c = 0; c < BT; ++c) y += sT[c * 65 + r] * sB2[c * LDT + jj];
        part += y * sB3[r * LDT + jj];
        if (r < bi.len) stf(dvo + ((size_t)(bi.tok0 + r) * H + h) * dv + j0 + jj, sb[r] * y);
      }
    }
    part = quad_sum(part);
    __syncthreads();
    if (q4 == 0) sdb[r] += part;
  }
  __syncthreads();
  if (tid == 0) {
    float rho = 0.f, hs = 0.f;
    for (int rr = 0; rr < BT; ++rr) rho += srho[rr];
    for (int w = 0; w < NT / 32; ++w) hs += sred[w];
    sdgam[BT - 1] += rho + expf(sg[BT - 1]) * hs;
    float acc = 0.f;
    for (int rr = BT - 1; rr >= 0; --rr) {
      acc += sdgam[rr];
      srho[rr] = acc;  // reuse: dg
    }
  }
  __syncthreads();
  if (r < bi.len) {
    const size_t tok = (size_t)(bi.tok0 + r) * H + h;
#pragma unroll
    for (int mi = 0; mi < NI; ++mi) {
      const int i = q4 + 4 * mi;
      stf(dq + tok * DK + i, aQ[mi]);
      stf(dk + tok * DK + i, aK[mi]);
    }
    if (q4 == 0) {
      stf(dg + tok, srho[r]);
      stf(dbeta + tok, sdb[r]);
    }
  }
}

// ---------------------------------------------------------------- launchers
constexpr size_t f4(size_t n) { return n * sizeof(float); }

template <int DK> size_t smem_pre() { return f4(BT * (DK + 1) + 3 * BT * 65 + 3 * BT); }
template <int DK> size_t smem_st() { return f4(2 * BT * (DK + 1) + DK * SBV + BT * SBV + BT); }
template <int DK> size_t smem_out() { return f4(2 * BT * (DK + 1) + BT * 65 + DK * 65 + BT * 65 + BT); }
template <int DK> size_t smem_st_bwd() {
  return f4(3 * BT * (DK + 1) + BT * 65 + DK * SBV + 2 * BT * SBV + BT);
}
template <int DK> size_t smem_grad() {
  return f4(3 * BT * (DK + 1) + 5 * BT * 65 + 2 * DK * (GT + 1) + 3 * BT * (GT + 1) + 7 * BT + NT / 32);
}

template <class K>
cudaError_t prep(K kernel, size_t smem) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <typename TI, int DK>
cudaError_t simt_fwd_t(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                       const void* g, const void* beta, const float* S_in, void* o,
                       float* S_out, const SimtWs& ws, cudaStream_t st) {
  const TI *Q = (const TI*)q, *K = (const TI*)k, *V = (const TI*)v, *G = (const TI*)g,
           *Bt = (const TI*)beta;
  cudaError_t e;
  if ((e = prep(k_pre<TI, DK>, smem_pre<DK>()))) return e;
  if ((e = prep(k_st<TI, DK>, smem_st<DK>()))) return e;
  if ((e = prep(k_out<TI, DK>, smem_out<DK>()))) return e;
  const dim3 gblk(m.nblk_cap, m.H);
  if (m.nblk_cap > 0) {
    prof_mark(st, "simt_pre");
    k_pre<TI, DK><<<gblk, NT, smem_pre<DK>(), st>>>(m, dv, K, V, G, Bt, ws);
  }
  prof_mark(st, "simt_st");
  k_st<TI, DK><<<m.nseq * m.H * (dv / SBV), NT, smem_st<DK>(), st>>>(m, dv, K, S_in, S_out, ws);
  if (m.nblk_cap > 0) {
    prof_mark(st, "simt_out");
    k_out<TI, DK><<<gblk, NT, smem_out<DK>(), st>>>(m, dv, Q, K, (TI*)o, ws);
  }
  prof_mark(st, nullptr);
  return cudaGetLastError();
}

template <typename TI, int DK>
cudaError_t simt_bwd_t(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                       const void* g, const void* beta, const float* S_in, const void* dout,
                       const float* dS_out, void* dq, void* dk, void* dvo, void* dg,
                       void* dbeta, float* dS_in, const SimtWs& ws, cudaStream_t st) {
  const TI *Q = (const TI*)q, *K = (const TI*)k, *V = (const TI*)v, *G = (const TI*)g,
           *Bt = (const TI*)beta, *dO = (const TI*)dout;
  cudaError_t e;
  if ((e = prep(k_pre<TI, DK>, smem_pre<DK>()))) return e;
  if ((e = prep(k_st<TI, DK>, smem_st<DK>()))) return e;
  if ((e = prep(k_st_bwd<TI, DK>, smem_st_bwd<DK>()))) return e;
  if ((e = prep(k_grad<TI, DK>, smem_grad<DK>()))) return e;
  const dim3 gblk(m.nblk_cap, m.H);
  const int nchain = m.nseq * m.H * (dv / SBV);
  if (m.nblk_cap > 0) {
    prof_mark(st, "simt_pre");
    k_pre<TI, DK><<<gblk, NT, smem_pre<DK>(), st>>>(m, dv, K, V, G, Bt, ws);
  }
  prof_mark(st, "simt_st");
  k_st<TI, DK><<<nchain, NT, smem_st<DK>(), st>>>(m, dv, K, S_in, nullptr, ws);
  prof_mark(st, "simt_st_bwd");
  k_st_bwd<TI, DK><<<nchain, NT, smem_st_bwd<DK>(), st>>>(m, dv, Q, K, dO, dS_out, dS_in, ws);
  if (m.nblk_cap > 0) {
    prof_mark(st, "simt_grad");
    k_grad<TI, DK><<<gblk, NT, smem_grad<DK>(), st>>>(m, dv, Q, K, V, Bt, dO, (TI*)dq, (TI*)dk,
                                                      (TI*)dvo, (TI*)dg, (TI*)dbeta, ws);
  }
  prof_mark(st, nullptr);
  return cudaGetLastError();
}

}  // namespace

size_t simt_max_smem() { return smem_grad<128>(); }

cudaError_t simt_fwd(const SeqMap& m, int dk, int dv, int dtype, const void* q, const void* k,
                     const void* v, const void* g, const void* beta, const float* S_in,
                     void* o, float* S_out, const SimtWs& ws, cudaStream_t st) {
  if (dtype == 0) {
    if (dk == 64) return simt_fwd_t<float, 64>(m, dv, q, k, v, g, beta, S_in, o, S_out, ws, st);
    return simt_fwd_t<float, 128>(m, dv, q, k, v, g, beta, S_in, o, S_out, ws, st);
  }
  if (dk == 64)
    return simt_fwd_t<__nv_bfloat16, 64>(m, dv, q, k, v, g, beta, S_in, o, S_out, ws, st);
  return simt_fwd_t<__nv_bfloat16, 128>(m, dv, q, k, v, g, beta, S_in, o, S_out, ws, st);
}

cudaError_t simt_bwd(const SeqMap& m, int dk, int dv, int dtype, const void* q, const void* k,
                     const void* v, const void* g, const void* beta, const float* S_in,
                     const void* dout, const float* dS_out, void* dq, void* dkk, void* dvv,
                     void* dg, void* dbeta, float* dS_in, const SimtWs& ws, cudaStream_t st) {
  if (dtype == 0) {
    if (dk == 64)
      return simt_bwd_t<float, 64>(m, dv, q, k, v, g, beta, S_in, dout, dS_out, dq, dkk, dvv, dg,
                                   dbeta, dS_in, ws, st);
    return simt_bwd_t<float, 128>(m, dv, q, k, v, g, beta, S_in, dout, dS_out, dq, dkk, dvv, dg,
                                  dbeta, dS_in, ws, st);
  }
  if (dk == 64)
    return simt_bwd_t<__nv_bfloat16, 64>(m, dv, q, k, v, g, beta, S_in, dout, dS_out, dq, dkk,
                                         dvv, dg, dbeta, dS_in, ws, st);
  return simt_bwd_t<__nv_bfloat16, 128>(m, dv, q, k, v, g, beta, S_in, dout, dS_out, dq, dkk,
                                        dvv, dg, dbeta, dS_in, ws, st);
}

}  // namespace gdn
