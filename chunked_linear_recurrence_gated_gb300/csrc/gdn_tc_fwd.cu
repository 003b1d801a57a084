// bf16 tensor-core kernels of the chunkwise gated delta rule: Pre and the
// register-resident ST chain fused with Out (forward), plus the chain's
// recompute mode used by the backward pass.
//
// Per 64-token block (StateFlow review: Pre / ST / Out with V^new, Eq. 2;
// kernel-level blocks b_{i,j}; tile size BV over the value dimension):
//   Pre : A = strictly-lower(diag(beta) K K^T * Mask), T = (I + A)^-1 (fp32),
//         W = T diag(beta Gamma) K, U = T diag(beta) V, QKM = Q K^T * Mask
//   ST  : V^new = U - W H_b ; H_{b+1} = Gamma_C H_b + K^T diag(e^{gamma_C - gamma}) V^new
//   Out : O = diag(Gamma) Q H_b + QKM V^new
// The state H is carried in fp32 registers as H^T (value rows, key columns)
// by the warps of one CTA per (sequence, head, 16 value columns); only its bf16
// copy feeds the tensor cores. All contractions are bf16 x bf16 -> fp32.
#include "gdn_internal.cuh"
#include "gdn_mma.cuh"

namespace gdn {
namespace {

constexpr int LDK = 136;   // padded smem row (bf16) for 128-wide tiles
constexpr int LD64 = 72;   // padded smem row (bf16) for 64-wide tiles

// ------------------------------------------------------------------ Pre
template <int DV>
struct PreSmem {
  __nv_bfloat16 K[BT * LDK];
  __nv_bfloat16 Q[BT * LDK];  // reused as the fp32 strictly-lower A (same size) after Q K^T
  __nv_bfloat16 V[BT * (DV + 8)];
  float Tf[BT * 68];    // T (fp32)
  float S[3 * 16 * 17]; // block products of the inverse
  __nv_bfloat16 T[BT * LD64];
  float g[BT];
  float b[BT];
  float bG[BT];
};

// Inclusive prefix sum of the 64 values in sg (warp 0), fixed order.
__device__ __forceinline__ void block_cumsum64(float* sg) {
  if (threadIdx.x < 32) {
    const int l = threadIdx.x;
    float a = sg[l], c = sg[l + 32];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float ya = __shfl_up_sync(0xffffffffu, a, off);
      const float yc = __shfl_up_sync(0xffffffffu, c, off);
      if (l >= off) {
        a += ya;
        c += yc;
      }
    }
    const float tot = __shfl_sync(0xffffffffu, a, 31);
    sg[l] = a;
    sg[l + 32] = c + tot;
  }
}

// T = (I + A)^-1 for strictly-lower 64 x 64 A (fp32, ld 68), 128 threads.
// Diagonal 16 x 16 blocks by forward substitution (one warp each), then block
// rows i = 1..3: T_ij = -T_ii sum_{m=j}^{i-1} A_im T_mj.
__device__ void invert_unit_lower64(const float* A, float* Tf, float* S) {
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  for (int idx = tid; idx < BT * 68; idx += 128) Tf[idx] = 0.f;
  __syncthreads();
  if (l < 16) {
    const int c = 16 * w + l;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float v = (r == l) ? 1.f : 0.f;
      const float* Ar = A + (16 * w + r) * 68 + 16 * w;
#pragma unroll
      for (int j = 0; j < r; ++j) v -= Ar[j] * x[j];
      x[r] = v;
      Tf[(16 * w + r) * 68 + c] = v;
    }
  }
  __syncthreads();
  for (int i = 1; i < 4; ++i) {
    // S_j = sum_{m=j}^{i-1} A_im T_mj for j < i
    for (int idx = tid; idx < i * 256; idx += 128) {
      const int j = idx >> 8, e = idx & 255, r = e >> 4, c = e & 15;
      float acc = 0.f;
      for (int m = j; m < i; ++m) {
        const float* Ar = A + (16 * i + r) * 68 + 16 * m;
        const float* Tc = Tf + (16 * m) * 68 + 16 * j + c;
#pragma unroll
        for (int q = 0; q < 16; ++q) acc += Ar[q] * Tc[q * 68];
      }
      S[j * 272 + r * 17 + c] = acc;
    }
    __syncthreads();
    for (int idx = tid; idx < i * 256; idx += 128) {
      const int j = idx >> 8, e = idx & 255, r = e >> 4, c = e & 15;
      const float* Tr = Tf + (16 * i + r) * 68 + 16 * i;
      float acc = 0.f;
      for (int q = 0; q <= r; ++q) acc += Tr[q] * S[j * 272 + q * 17 + c];
      Tf[(16 * i + r) * 68 + 16 * j + c] = -acc;
    }
    __syncthreads();
  }
}

template <int DV>
__global__ void __launch_bounds__(128) k_pre_tc(SeqMap m, const __nv_bfloat16* __restrict__ q,
                                                const __nv_bfloat16* __restrict__ k,
                                                const __nv_bfloat16* __restrict__ v,
                                                const __nv_bfloat16* __restrict__ g,
                                                const __nv_bfloat16* __restrict__ beta,
                                                TcWs ws) {
  constexpr int DK = 128;
  constexpr int LDV = DV + 8;
  BlockInfo bi;
  const int gb = blockIdx.x, h = blockIdx.y, H = m.H, tid = threadIdx.x;
  if (!block_info(m, gb, bi)) return;
  extern __shared__ __align__(16) unsigned char smraw[];
  PreSmem<DV>& sm = *reinterpret_cast<PreSmem<DV>*>(smraw);
  const int w = tid >> 5, l = tid & 31, gq = l >> 2, tq = l & 3;
  const size_t bh = (size_t)gb * H + h;

  // loads (rows past the block's end are zero-filled)
  for (int idx = tid; idx < BT * (DK / 8); idx += 128) {
    const int r = idx >> 4, c = (idx & 15) * 8;
    const bool ok = r < bi.len;
    const size_t off = ((size_t)(bi.tok0 + (ok ? r : 0)) * H + h) * DK + c;
    cp16(&sm.K[r * LDK + c], k + off, ok);
    cp16(&sm.Q[r * LDK + c], q + off, ok);
  }
  for (int idx = tid; idx < BT * (DV / 8); idx += 128) {
    const int r = idx / (DV / 8), c = (idx % (DV / 8)) * 8;
    const bool ok = r < bi.len;
    cp16(&sm.V[r * LDV + c], v + ((size_t)(bi.tok0 + (ok ? r : 0)) * H + h) * DV + c, ok);
  }
  cp_commit();
  if (tid < BT) {
    const bool ok = tid < bi.len;
    const size_t off = (size_t)(bi.tok0 + tid) * H + h;
    sm.g[tid] = ok ? __bfloat162float(g[off]) : 0.f;
    sm.b[tid] = ok ? __bfloat162float(beta[off]) : 0.f;
  }
  __syncthreads();
  block_cumsum64(sm.g);
  cp_wait<0>();
  __syncthreads();
  if (tid < BT) {
    sm.bG[tid] = sm.b[tid] * expf(sm.g[tid]);
    ws.gam[bh * BT + tid] = sm.g[tid];
  }

  // K K^T and Q K^T, rows [16w, 16w + 16)
  {
    float kk[8][4], qk[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) kk[j][e] = qk[j][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < DK / 16; ++kc) {
      uint32_t ak[4], aq[4];
      lda_rm(ak, sm.K, LDK, 16 * w, 16 * kc);
      lda_rm(aq, sm.Q, LDK, 16 * w, 16 * kc);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        uint32_t b[4];
        ldb_nk_x2n(b, sm.K, LDK, 16 * jj, 16 * kc);
        mma16816(kk[2 * jj], ak, b[0], b[1]);
        mma16816(kk[2 * jj + 1], ak, b[2], b[3]);
        mma16816(qk[2 * jj], aq, b[0], b[1]);
        mma16816(qk[2 * jj + 1], aq, b[2], b[3]);
      }
    }
    __nv_bfloat16* qkm = ws.QKM + bh * BT * BT;
    float* sA = reinterpret_cast<float*>(sm.Q);
    __syncthreads();  // every warp is done reading Q before A overwrites it
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = 16 * w + gq + 8 * hf;
        const int c = 8 * j + 2 * tq;
        const float gr = sm.g[r];
        const float d0 = expf(gr - sm.g[c]), d1 = expf(gr - sm.g[c + 1]);
        const float br = sm.b[r];
        sA[r * 68 + c] = (c < r) ? br * kk[j][2 * hf] * d0 : 0.f;
        sA[r * 68 + c + 1] = (c + 1 < r) ? br * kk[j][2 * hf + 1] * d1 : 0.f;
        const float m0 = (c <= r) ? qk[j][2 * hf] * d0 : 0.f;
        const float m1 = (c + 1 <= r) ? qk[j][2 * hf + 1] * d1 : 0.f;
        *reinterpret_cast<uint32_t*>(qkm + r * BT + c) = pack_bf16(m0, m1);
      }
  }
  __syncthreads();
  invert_unit_lower64(reinterpret_cast<const float*>(sm.Q), sm.Tf, sm.S);
  // T -> bf16; K <- diag(beta Gamma) K ; V <- diag(beta) V
  for (int idx = tid; idx < BT * BT; idx += 128) {
    const int r = idx >> 6, c = idx & 63;
    const __nv_bfloat16 t = __float2bfloat16_rn(sm.Tf[r * 68 + c]);
    sm.T[r * LD64 + c] = t;
    if (ws.T) ws.T[bh * BT * BT + idx] = t;
  }
  for (int idx = tid; idx < BT * DK; idx += 128) {
    const int r = idx >> 7, c = idx & 127;
    sm.K[r * LDK + c] = __float2bfloat16_rn(__bfloat162float(sm.K[r * LDK + c]) * sm.bG[r]);
  }
  for (int idx = tid; idx < BT * DV; idx += 128) {
    const int r = idx / DV, c = idx % DV;
    sm.V[r * LDV + c] = __float2bfloat16_rn(__bfloat162float(sm.V[r * LDV + c]) * sm.b[r]);
  }
  __syncthreads();
  uint32_t at[4][4];
#pragma unroll
  for (int kc = 0; kc < 4; ++kc) lda_rm(at[kc], sm.T, LD64, 16 * w, 16 * kc);
  // W = T (beta Gamma K): rows [16w, 16w+16), 128 columns
  {
    float acc[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < 4; ++kc)
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        uint32_t b[4];
        ldb_kn_x2n(b, sm.K, LDK, 16 * kc, 16 * jj);
        mma16816(acc[2 * jj], at[kc], b[0], b[1]);
        mma16816(acc[2 * jj + 1], at[kc], b[2], b[3]);
      }
    __nv_bfloat16* W = ws.W + bh * BT * DK;
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = 16 * w + gq + 8 * hf, c = 8 * j + 2 * tq;
        *reinterpret_cast<uint32_t*>(W + r * DK + c) = pack_bf16(acc[j][2 * hf], acc[j][2 * hf + 1]);
      }
  }
  // U = T (beta V), 128 columns at a time; stored tile-major [DV/16][64][16]
#pragma unroll
  for (int c0 = 0; c0 < DV; c0 += 128) {
    float acc[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < 4; ++kc)
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        uint32_t b[4];
        ldb_kn_x2n(b, sm.V, LDV, 16 * kc, c0 + 16 * jj);
        mma16816(acc[2 * jj], at[kc], b[0], b[1]);
        mma16816(acc[2 * jj + 1], at[kc], b[2], b[3]);
      }
    __nv_bfloat16* U = ws.U + bh * BT * DV;
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = 16 * w + gq + 8 * hf, c = c0 + 8 * j + 2 * tq;
        *reinterpret_cast<uint32_t*>(U + (c >> 4) * BT * 16 + r * 16 + (c & 15)) =
            pack_bf16(acc[j][2 * hf], acc[j][2 * hf + 1]);
      }
  }
}

// ------------------------------------------------------------------ ST chain (+ Out)
// One CTA per (sequence, head, 16 value columns), 4 warps, sequential over the
// sequence's 64-token blocks. Warp w owns key columns [32w, 32w + 32) of the
// fp32 state H^T (16 x 128) and tokens [16w, 16w + 16) of each block's V^new
// and O. Per block:
//   X^T   = H^T W^T                       (tokens of warp w, K = 128)
//   V^newT = U^T - X^T ;  Vs^T = V^newT * e^{gamma_C - gamma}
//   H^T  <- Gamma_C H^T + Vs^T K           (key columns of warp w, K = 64)
//   O^T   = (H^T Q^T) * Gamma + V^newT QKM^T (FWD)
// The bf16 copies of H^T and V^new^T are exchanged through shared memory.
constexpr int NSTAGE = 3;
enum { CHAIN_FWD = 0, CHAIN_RECOMPUTE = 1 };

template <int MODE>
struct ChainStage {
  __nv_bfloat16 W[BT * LDK];
  __nv_bfloat16 K[BT * LDK];
  __nv_bfloat16 Q[MODE == CHAIN_FWD ? BT * LDK : 8];
  __nv_bfloat16 QKM[MODE == CHAIN_FWD ? BT * LD64 : 8];
  __nv_bfloat16 U[BT * 24];
  float g[BT];
};

template <int MODE>
struct ChainSmem {
  ChainStage<MODE> st[NSTAGE];
  __nv_bfloat16 HT[16 * LDK];
  __nv_bfloat16 VnT[16 * LD64];
  __nv_bfloat16 VsT[16 * LD64];
  __nv_bfloat16 O[BT * 24];
};

template <int DV, int MODE>
__global__ void __launch_bounds__(128, 1) k_chain(SeqMap m, const __nv_bfloat16* __restrict__ q,
                                                  const __nv_bfloat16* __restrict__ k,
                                                  const float* S_in, float* S_out,
                                                  __nv_bfloat16* __restrict__ o, TcWs ws) {
  constexpr int DK = 128;
  constexpr int NVT = DV / 16;
  const int tile = blockIdx.x % NVT;
  const int sh = blockIdx.x / NVT;
  const int H = m.H, h = sh % H, s = sh / H;
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31, gq = l >> 2, tq = l & 3;
  if (m.cu == nullptr && blockIdx.x == 0 && tid == 0) ws.status[0] = DEV_OK;
  const SeqInfo si = seq_info(m, s);
  extern __shared__ __align__(16) unsigned char smraw[];
  ChainSmem<MODE>& sm = *reinterpret_cast<ChainSmem<MODE>*>(smraw);

  // fp32 state slice: H^T rows v = gq (+8), key columns 32w + 8j + 2tq (+1)
  float hs[4][4];
  const size_t sbase = ((size_t)s * H + h) * DK * DV + (size_t)tile * 16;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int vr = gq + 8 * (e >> 1);
      const int kc = 32 * w + 8 * j + 2 * tq + (e & 1);
      hs[j][e] = S_in ? S_in[sbase + (size_t)kc * DV + vr] : 0.f;
    }
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int vr = gq + 8 * hf, kc = 32 * w + 8 * j + 2 * tq;
      *reinterpret_cast<uint32_t*>(&sm.HT[vr * LDK + kc]) = pack_bf16(hs[j][2 * hf], hs[j][2 * hf + 1]);
    }

  auto load_block = [&](int lb) {
    ChainStage<MODE>& S = sm.st[lb % NSTAGE];
    const int gb = si.blk0 + lb, tok0 = si.tok0 + lb * BT, len = min(BT, si.len - lb * BT);
    const size_t bh = (size_t)gb * H + h;
    const __nv_bfloat16* Wg = ws.W + bh * BT * DK;
    for (int idx = tid; idx < BT * 16; idx += 128) {
      const int r = idx >> 4, c = (idx & 15) * 8;
      const bool ok = r < len;
      const size_t off = ((size_t)(tok0 + (ok ? r : 0)) * H + h) * DK + c;
      cp16(&S.W[r * LDK + c], Wg + r * DK + c, true);
      cp16(&S.K[r * LDK + c], k + off, ok);
      if (MODE == CHAIN_FWD) cp16(&S.Q[r * LDK + c], q + off, ok);
    }
    if (MODE == CHAIN_FWD) {
      const __nv_bfloat16* Mg = ws.QKM + bh * BT * BT;
      for (int idx = tid; idx < BT * 8; idx += 128) {
        const int r = idx >> 3, c = (idx & 7) * 8;
        cp16(&S.QKM[r * LD64 + c], Mg + r * BT + c, true);
      }
    }
    {
      const __nv_bfloat16* Ug = ws.U + bh * BT * DV + (size_t)tile * BT * 16;
      const int r = tid >> 1, c = (tid & 1) * 8;
      cp16(&S.U[r * 24 + c], Ug + r * 16 + c, true);
    }
    if (tid < 16) cp16(&S.g[tid * 4], ws.gam + bh * BT + tid * 4, true);
  };

#pragma unroll
  for (int i = 0; i < NSTAGE - 1; ++i) {
    if (i < si.nblk) load_block(i);
    cp_commit();
  }

  for (int lb = 0; lb < si.nblk; ++lb) {
    cp_wait<NSTAGE - 2>();
    __syncthreads();
    if (lb + NSTAGE - 1 < si.nblk) load_block(lb + NSTAGE - 1);
    cp_commit();
    const ChainStage<MODE>& S = sm.st[lb % NSTAGE];
    const int gb = si.blk0 + lb, tok0 = si.tok0 + lb * BT, len = min(BT, si.len - lb * BT);
    const size_t bh = (size_t)gb * H + h;
    const float gC = S.g[BT - 1];

    if (MODE == CHAIN_RECOMPUTE) {
      // H_b (bf16, value-major) for the backward kernels
      __nv_bfloat16* Hg = ws.HbT + bh * DV * DK + (size_t)tile * 16 * DK;
      for (int idx = tid; idx < 16 * 16; idx += 128) {
        const int r = idx >> 4, c = (idx & 15) * 8;
        *reinterpret_cast<uint4*>(Hg + r * DK + c) = *reinterpret_cast<const uint4*>(&sm.HT[r * LDK + c]);
      }
    }

    // X^T = H^T W^T (and H^T Q^T) for tokens [16w, 16w + 16)
    float x[2][4], o1[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[j][e] = o1[j][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < DK / 16; ++kc) {
      uint32_t a[4], b[4];
      lda_rm(a, sm.HT, LDK, 0, 16 * kc);
      ldb_nk_x2n(b, S.W, LDK, 16 * w, 16 * kc);
      mma16816(x[0], a, b[0], b[1]);
      mma16816(x[1], a, b[2], b[3]);
      if (MODE == CHAIN_FWD) {
        ldb_nk_x2n(b, S.Q, LDK, 16 * w, 16 * kc);
        mma16816(o1[0], a, b[0], b[1]);
        mma16816(o1[1], a, b[2], b[3]);
      }
    }
    // V^new^T = U^T - X^T ; scaled copy for the state update
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int vr = gq + 8 * hf;
        const int t0 = 16 * w + 8 * j + 2 * tq;
        const float u0 = __bfloat162float(S.U[t0 * 24 + vr]);
        const float u1 = __bfloat162float(S.U[(t0 + 1) * 24 + vr]);
        const float v0 = u0 - x[j][2 * hf], v1 = u1 - x[j][2 * hf + 1];
        const float s0 = v0 * expf(gC - S.g[t0]), s1 = v1 * expf(gC - S.g[t0 + 1]);
        const uint32_t pv = pack_bf16(v0, v1);
        *reinterpret_cast<uint32_t*>(&sm.VnT[vr * LD64 + t0]) = pv;
        *reinterpret_cast<uint32_t*>(&sm.VsT[vr * LD64 + t0]) = pack_bf16(s0, s1);
        if (MODE == CHAIN_RECOMPUTE)
          *reinterpret_cast<uint32_t*>(ws.VnT + bh * DV * BT + (size_t)(tile * 16 + vr) * BT + t0) = pv;
      }
    __syncthreads();

    // H^T <- Gamma_C H^T + Vs^T K on key columns [32w, 32w + 32)
    const float GC = expf(gC);
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) hs[j][e] *= GC;
    float o2[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) o2[j][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
      uint32_t a[4], b[4];
      lda_rm(a, sm.VsT, LD64, 0, 16 * kc);
      ldb_kn_x2n(b, S.K, LDK, 16 * kc, 32 * w);
      mma16816(hs[0], a, b[0], b[1]);
      mma16816(hs[1], a, b[2], b[3]);
      ldb_kn_x2n(b, S.K, LDK, 16 * kc, 32 * w + 16);
      mma16816(hs[2], a, b[0], b[1]);
      mma16816(hs[3], a, b[2], b[3]);
      if (MODE == CHAIN_FWD) {
        lda_rm(a, sm.VnT, LD64, 0, 16 * kc);
        ldb_nk_x2n(b, S.QKM, LD64, 16 * w, 16 * kc);
        mma16816(o2[0], a, b[0], b[1]);
        mma16816(o2[1], a, b[2], b[3]);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int vr = gq + 8 * hf, kc = 32 * w + 8 * j + 2 * tq;
        *reinterpret_cast<uint32_t*>(&sm.HT[vr * LDK + kc]) = pack_bf16(hs[j][2 * hf], hs[j][2 * hf + 1]);
      }
    if (MODE == CHAIN_FWD) {
      // O[token][v] = Gamma_token (H^T Q^T)^T + (V^new^T QKM^T)^T, staged for coalesced stores
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int vr = gq + 8 * (e >> 1);
          const int t = 16 * w + 8 * j + 2 * tq + (e & 1);
          sm.O[t * 24 + vr] = __float2bfloat16_rn(expf(S.g[t]) * o1[j][e] + o2[j][e]);
        }
      __syncwarp();
      // each warp stores its own 16 tokens (16 rows x 32 bytes)
      {
        const int r = 16 * w + (l >> 1), c = (l & 1) * 8;
        if (r < len)
          *reinterpret_cast<uint4*>(o + ((size_t)(tok0 + r) * H + h) * DV + tile * 16 + c) =
              *reinterpret_cast<const uint4*>(&sm.O[r * 24 + c]);
      }
    }
  }
  if (S_out) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int vr = gq + 8 * (e >> 1);
        const int kc = 32 * w + 8 * j + 2 * tq + (e & 1);
        S_out[sbase + (size_t)kc * DV + vr] = hs[j][e];
      }
  }
}

template <class K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int DV>
cudaError_t tc_fwd_t(const SeqMap& m, const void* q, const void* k, const void* v, const void* g,
                     const void* beta, const float* S_in, void* o, float* S_out, const TcWs& ws,
                     cudaStream_t st) {
  using bf = __nv_bfloat16;
  cudaError_t e;
  if ((e = set_smem(k_pre_tc<DV>, sizeof(PreSmem<DV>)))) return e;
  if ((e = set_smem(k_chain<DV, CHAIN_FWD>, sizeof(ChainSmem<CHAIN_FWD>)))) return e;
  if (m.nblk_cap > 0) {
    prof_mark(st, "tc_pre");
    k_pre_tc<DV><<<dim3(m.nblk_cap, m.H), 128, sizeof(PreSmem<DV>), st>>>(
        m, (const bf*)q, (const bf*)k, (const bf*)v, (const bf*)g, (const bf*)beta, ws);
  }
  prof_mark(st, "tc_chain_fwd");
  k_chain<DV, CHAIN_FWD><<<m.nseq * m.H * (DV / 16), 128, sizeof(ChainSmem<CHAIN_FWD>), st>>>(
      m, (const bf*)q, (const bf*)k, S_in, S_out, (bf*)o, ws);
  prof_mark(st, nullptr);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_fwd(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const float* S_in, void* o, float* S_out,
                   const TcWs& ws, cudaStream_t st) {
  if (dv == 128) return tc_fwd_t<128>(m, q, k, v, g, beta, S_in, o, S_out, ws, st);
  return tc_fwd_t<256>(m, q, k, v, g, beta, S_in, o, S_out, ws, st);
}

// Pre + recompute chain for the backward pass (W, U, QKM, T, gamma, H_b, V^new).
cudaError_t tc_bwd_prep(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                        const void* g, const void* beta, const float* S_in, const TcWs& ws,
                        cudaStream_t st) {
  using bf = __nv_bfloat16;
  cudaError_t e;
  if (dv == 128) {
    if ((e = set_smem(k_pre_tc<128>, sizeof(PreSmem<128>)))) return e;
    if ((e = set_smem(k_chain<128, CHAIN_RECOMPUTE>, sizeof(ChainSmem<CHAIN_RECOMPUTE>)))) return e;
  } else {
    if ((e = set_smem(k_pre_tc<256>, sizeof(PreSmem<256>)))) return e;
    if ((e = set_smem(k_chain<256, CHAIN_RECOMPUTE>, sizeof(ChainSmem<CHAIN_RECOMPUTE>)))) return e;
  }
  if (m.nblk_cap > 0) {
    prof_mark(st, "tc_pre");
    if (dv == 128)
      k_pre_tc<128><<<dim3(m.nblk_cap, m.H), 128, sizeof(PreSmem<128>), st>>>(
          m, (const bf*)q, (const bf*)k, (const bf*)v, (const bf*)g, (const bf*)beta, ws);
    else
      k_pre_tc<256><<<dim3(m.nblk_cap, m.H), 128, sizeof(PreSmem<256>), st>>>(
          m, (const bf*)q, (const bf*)k, (const bf*)v, (const bf*)g, (const bf*)beta, ws);
  }
  prof_mark(st, "tc_chain_recompute");
  const int grid = m.nseq * m.H * (dv / 16);
  if (dv == 128)
    k_chain<128, CHAIN_RECOMPUTE><<<grid, 128, sizeof(ChainSmem<CHAIN_RECOMPUTE>), st>>>(
        m, (const bf*)q, (const bf*)k, S_in, nullptr, nullptr, ws);
  else
    k_chain<256, CHAIN_RECOMPUTE><<<grid, 128, sizeof(ChainSmem<CHAIN_RECOMPUTE>), st>>>(
        m, (const bf*)q, (const bf*)k, S_in, nullptr, nullptr, ws);
  return cudaGetLastError();
}

}  // namespace gdn
