// Pre kernel of the bf16 tensor-core path: per 64-token block and head, the
// WY factors and masks every later step reads.
//
// Per 64-token block (StateFlow review: Pre / ST / Out with V^new, Eq. 2;
// kernel-level blocks b_{i,j}; tile size BV over the value dimension):
//   Pre : A = strictly-lower(diag(beta) K K^T * Mask), T = (I + A)^-1 (fp32),
//         W = T diag(beta Gamma) K, U = T diag(beta) V, QKM = Q K^T * Mask
//   ST  : V^new = U - W H_b ; H_{b+1} = Gamma_C H_b + K^T diag(e^{gamma_C - gamma}) V^new
//   Out : O = diag(Gamma) Q H_b + QKM V^new
// Pre also writes padded, decay-scaled copies of the block's rows,
// K~ = diag(e^{gamma_C - gamma}) K and Q~ = diag(e^{gamma}) Q, and the per-row
// vectors (Gamma_r, e^{gamma_C - gamma_r}, gamma_r, beta_r), so that the
// sequential chains fetch every operand with one bulk copy and scale nothing
// but the state. All contractions are bf16 x bf16 -> fp32 warp-level MMAs;
// the triangular inverse is fp32 with TF32 MMAs for its off-diagonal blocks.
#include "gdn_internal.cuh"
#include "gdn_mma.cuh"

namespace gdn {
namespace {

constexpr int LDK = TC_LDK;
constexpr int LD64 = TC_LD64;
constexpr int LDU = TC_LDU;

// ------------------------------------------------------------------ Pre
template <int DV>
struct PreSmem {
  __nv_bfloat16 K[BT * LDK];
  __nv_bfloat16 Q[BT * LDK];  // reused as the fp32 strictly-lower A (same size) after Q K^T
  __nv_bfloat16 V[BT * (DV + 8)];
  float Tf[BT * 68];          // T (fp32)
  float S[16 * 52];           // block-row product of the inverse
  __nv_bfloat16 Tw[BT * LD64];  // T diag(beta Gamma)
  __nv_bfloat16 Tu[BT * LD64];  // T diag(beta)
  float g[BT];
  float b[BT];
  float G[BT];
  float dte[BT];
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

// T = (I + A)^-1 for strictly-lower 64 x 64 A (fp32, ld 68), NT threads.
// The four diagonal 16 x 16 blocks by fp32 forward substitution (one warp
// each); then, block row by block row (i = 1..3), warps 0..2i-1 (one n8
// column tile each) form
//   S = A[i, 0:i] T[0:i, 0:i]   and   T[i, 0:i] = -T_ii S
// with TF32 tensor-core MMAs (fp32 accumulation): the block products of
// T_ij = -T_ii sum_{m=j}^{i-1} A_im T_mj for all j < i at once.
template <int NT>
__device__ void invert_unit_lower64(const float* A, float* Tf, float* S) {
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31, g = l >> 2, t = l & 3;
  for (int idx = tid; idx < BT * 68; idx += NT) Tf[idx] = 0.f;
  __syncthreads();
  if (w < 4 && l < 16) {
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
  // block row i: warp w < 2i owns the n8 column tile w of both products, so the
  // two products of a level need no barrier between them (each warp reads back
  // only its own S columns); one barrier per level publishes the new rows.
#pragma unroll
  for (int i = 1; i < 4; ++i) {
    const int R = 16 * i;
    if (w < 2 * i) {
      const int nt = w;
      // S (16 x 8, column tile nt) = A[R:R+16, 0:16i] * Tf[0:16i, 8nt:8nt+8]; fp32, ld 52
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int kt = 0; kt < 2 * i; ++kt) {
        uint32_t a[4];
        a[0] = to_tf32(A[(R + g) * 68 + 8 * kt + t]);
        a[1] = to_tf32(A[(R + g + 8) * 68 + 8 * kt + t]);
        a[2] = to_tf32(A[(R + g) * 68 + 8 * kt + t + 4]);
        a[3] = to_tf32(A[(R + g + 8) * 68 + 8 * kt + t + 4]);
        const uint32_t b0 = to_tf32(Tf[(8 * kt + t) * 68 + 8 * nt + g]);
        const uint32_t b1 = to_tf32(Tf[(8 * kt + t + 4) * 68 + 8 * nt + g]);
        mma_tf32(acc, a, b0, b1);
      }
      S[g * 52 + 8 * nt + 2 * t] = acc[0];
      S[g * 52 + 8 * nt + 2 * t + 1] = acc[1];
      S[(g + 8) * 52 + 8 * nt + 2 * t] = acc[2];
      S[(g + 8) * 52 + 8 * nt + 2 * t + 1] = acc[3];
      __syncwarp();
      // T[R:R+16, 8nt:8nt+8] = -T_ii S
      float acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kt = 0; kt < 2; ++kt) {
        uint32_t a[4];
        a[0] = to_tf32(Tf[(R + g) * 68 + R + 8 * kt + t]);
        a[1] = to_tf32(Tf[(R + g + 8) * 68 + R + 8 * kt + t]);
        a[2] = to_tf32(Tf[(R + g) * 68 + R + 8 * kt + t + 4]);
        a[3] = to_tf32(Tf[(R + g + 8) * 68 + R + 8 * kt + t + 4]);
        const uint32_t b0 = to_tf32(S[(8 * kt + t) * 52 + 8 * nt + g]);
        const uint32_t b1 = to_tf32(S[(8 * kt + t + 4) * 52 + 8 * nt + g]);
        mma_tf32(acc2, a, b0, b1);
      }
      Tf[(R + g) * 68 + 8 * nt + 2 * t] = -acc2[0];
      Tf[(R + g) * 68 + 8 * nt + 2 * t + 1] = -acc2[1];
      Tf[(R + g + 8) * 68 + 8 * nt + 2 * t] = -acc2[2];
      Tf[(R + g + 8) * 68 + 8 * nt + 2 * t + 1] = -acc2[3];
    }
    __syncthreads();
  }
}

// 8 warps; warp (rw = w & 3, cw = w >> 2) owns rows [16 rw, 16 rw + 16) and
// the cw-th half of the columns of every product.
template <int DV>
__global__ void __launch_bounds__(256, 2) k_pre_tc(SeqMap m, const __nv_bfloat16* __restrict__ q,
                                                   const __nv_bfloat16* __restrict__ k,
                                                   const __nv_bfloat16* __restrict__ v,
                                                   const __nv_bfloat16* __restrict__ g,
                                                   const __nv_bfloat16* __restrict__ beta,
                                                   TcWs ws) {
  constexpr int DK = 128;
  constexpr int LDV = DV + 8;
  constexpr int NT = 256;
  BlockInfo bi;
  const int gb = blockIdx.x, h = blockIdx.y, H = m.H, tid = threadIdx.x;
  // Pre is the first kernel of a fixed-length call: it clears the status word,
  // which the later kernels of the call only ever set (varlen calls: the
  // block-table kernel sets it)
  if (m.cu == nullptr && gb == 0 && h == 0 && tid == 0) ws.status[0] = DEV_OK;
  if (!block_info(m, gb, bi)) return;
  extern __shared__ __align__(128) unsigned char smraw[];
  PreSmem<DV>& sm = *reinterpret_cast<PreSmem<DV>*>(smraw);
  const int w = tid >> 5, l = tid & 31, gq = l >> 2, tq = l & 3;
  const int rw = w & 3, cw = w >> 2, R0 = 16 * rw;
  const size_t bh = (size_t)gb * H + h;

  for (int idx = tid; idx < BT * (DK / 8); idx += NT) {
    const int r = idx >> 4, c = (idx & 15) * 8;
    const bool ok = r < bi.len;
    const size_t off = ((size_t)(bi.tok0 + (ok ? r : 0)) * H + h) * DK + c;
    cp16(&sm.K[r * LDK + c], k + off, ok);
    cp16(&sm.Q[r * LDK + c], q + off, ok);
  }
  for (int idx = tid; idx < BT * (DV / 8); idx += NT) {
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
    const float gr = sm.g[tid];
    const float G = __expf(gr), dte = __expf(sm.g[BT - 1] - gr);
    sm.G[tid] = G;
    sm.dte[tid] = dte;
    float* dec = ws.dec + bh * TC_DEC_ROWS * BT;
    dec[tid] = G;
    dec[BT + tid] = dte;
    dec[2 * BT + tid] = gr;
    dec[3 * BT + tid] = sm.b[tid];
  }
  __syncthreads();
  // padded, decay-scaled copies for the chains (one bulk copy each per block):
  // K~ = diag(e^{gamma_C - gamma}) K and Q~ = diag(e^{gamma}) Q
  {
    const uint4* sK = reinterpret_cast<const uint4*>(sm.K);
    const uint4* sQ = reinterpret_cast<const uint4*>(sm.Q);
    uint4* gK = reinterpret_cast<uint4*>(ws.Kp + bh * BT * LDK);
    uint4* gQ = reinterpret_cast<uint4*>(ws.Qp + bh * BT * LDK);
    for (int idx = tid; idx < BT * LDK / 8; idx += NT) {
      const int r = idx / (LDK / 8);
      const float sk = sm.dte[r], sq = sm.G[r];
      uint4 a = sK[idx], b = sQ[idx];
      uint32_t* pa = &a.x;
      uint32_t* pb = &b.x;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = unpack_bf16(pa[e]), y = unpack_bf16(pb[e]);
        pa[e] = pack_bf16(sk * x.x, sk * x.y);
        pb[e] = pack_bf16(sq * y.x, sq * y.y);
      }
      gK[idx] = a;
      gQ[idx] = b;
    }
  }

  // K K^T and Q K^T on rows [R0, R0 + 16), columns [32 cw, 32 cw + 32)
  {
    float kk[4][4], qk[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) kk[j][e] = qk[j][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < DK / 16; ++kc) {
      uint32_t ak[4], aq[4];
      lda_rm(ak, sm.K, LDK, R0, 16 * kc);
      lda_rm(aq, sm.Q, LDK, R0, 16 * kc);
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        uint32_t b[4];
        ldb_nk_x2n(b, sm.K, LDK, 32 * cw + 16 * jj, 16 * kc);
        mma16816(kk[2 * jj], ak, b[0], b[1]);
        mma16816(kk[2 * jj + 1], ak, b[2], b[3]);
        mma16816(qk[2 * jj], aq, b[0], b[1]);
        mma16816(qk[2 * jj + 1], aq, b[2], b[3]);
      }
    }
    __nv_bfloat16* qkm = ws.QKM + bh * BT * LD64;
    float* sA = reinterpret_cast<float*>(sm.Q);
    __syncthreads();  // every warp is done reading Q before A overwrites it
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = R0 + gq + 8 * hf;
        const int c = 32 * cw + 8 * j + 2 * tq;
        const float gr = sm.g[r];
        const float d0 = (c <= r) ? __expf(gr - sm.g[c]) : 0.f;
        const float d1 = (c + 1 <= r) ? __expf(gr - sm.g[c + 1]) : 0.f;
        const float br = sm.b[r];
        const float km0 = (c < r) ? kk[j][2 * hf] * d0 : 0.f;
        const float km1 = (c + 1 < r) ? kk[j][2 * hf + 1] * d1 : 0.f;
        sA[r * 68 + c] = br * km0;
        sA[r * 68 + c + 1] = br * km1;
        if (ws.KKM)
          *reinterpret_cast<uint32_t*>(ws.KKM + bh * BT * LD64 + r * LD64 + c) = pack_bf16(km0, km1);
        *reinterpret_cast<uint32_t*>(qkm + r * LD64 + c) =
            pack_bf16(qk[j][2 * hf] * d0, qk[j][2 * hf + 1] * d1);
      }
  }
  __syncthreads();
  invert_unit_lower64<NT>(reinterpret_cast<const float*>(sm.Q), sm.Tf, sm.S);
  // Tw = T diag(beta Gamma), Tu = T diag(beta) (bf16); T itself for the backward
  for (int idx = 2 * tid; idx < BT * BT; idx += 2 * NT) {  // column pairs
    const int r = idx >> 6, c = idx & 63;
    const float2 t = *reinterpret_cast<const float2*>(&sm.Tf[r * 68 + c]);
    const float2 bc = *reinterpret_cast<const float2*>(&sm.b[c]);
    const float2 Gc = *reinterpret_cast<const float2*>(&sm.G[c]);
    *reinterpret_cast<uint32_t*>(&sm.Tw[r * LD64 + c]) =
        pack_bf16(t.x * bc.x * Gc.x, t.y * bc.y * Gc.y);
    *reinterpret_cast<uint32_t*>(&sm.Tu[r * LD64 + c]) = pack_bf16(t.x * bc.x, t.y * bc.y);
    if (ws.T) *reinterpret_cast<uint32_t*>(ws.T + bh * BT * BT + idx) = pack_bf16(t.x, t.y);
  }
  __syncthreads();
  // W = Tw K: rows [R0, R0 + 16), columns [64 cw, 64 cw + 64)
  {
    uint32_t at[4][4];
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) lda_rm(at[kc], sm.Tw, LD64, R0, 16 * kc);
    float acc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < 4; ++kc)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        uint32_t b[4];
        ldb_kn_x2n(b, sm.K, LDK, 16 * kc, 64 * cw + 16 * jj);
        mma16816(acc[2 * jj], at[kc], b[0], b[1]);
        mma16816(acc[2 * jj + 1], at[kc], b[2], b[3]);
      }
    __nv_bfloat16* W = ws.W + bh * BT * LDK;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = R0 + gq + 8 * hf, c = 64 * cw + 8 * j + 2 * tq;
        *reinterpret_cast<uint32_t*>(W + r * LDK + c) = pack_bf16(acc[j][2 * hf], acc[j][2 * hf + 1]);
      }
  }
  // U = Tu V: rows [R0, R0 + 16), columns [DV/2 cw, DV/2 (cw + 1)), 64 at a time
  {
    uint32_t at[4][4];
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) lda_rm(at[kc], sm.Tu, LD64, R0, 16 * kc);
    __nv_bfloat16* U = ws.U + bh * (DV / 16) * BT * LDU;
#pragma unroll
    for (int c0 = 0; c0 < DV / 2; c0 += 64) {
      const int cb = cw * (DV / 2) + c0;
      float acc[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
#pragma unroll
      for (int kc = 0; kc < 4; ++kc)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          uint32_t b[4];
          ldb_kn_x2n(b, sm.V, LDV, 16 * kc, cb + 16 * jj);
          mma16816(acc[2 * jj], at[kc], b[0], b[1]);
          mma16816(acc[2 * jj + 1], at[kc], b[2], b[3]);
        }
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int r = R0 + gq + 8 * hf, c = cb + 8 * j + 2 * tq;
          *reinterpret_cast<uint32_t*>(U + ((c >> 4) * BT + r) * LDU + (c & 15)) =
              pack_bf16(acc[j][2 * hf], acc[j][2 * hf + 1]);
        }
    }
  }
  // zero the pad columns of the padded tiles: every 32-byte sector is then
  // written in full, so none has to be read back from DRAM to merge it
  {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    __nv_bfloat16* W = ws.W + bh * BT * LDK;
    __nv_bfloat16* qkm = ws.QKM + bh * BT * LD64;
    __nv_bfloat16* U = ws.U + bh * (DV / 16) * BT * LDU;
    for (int r = tid; r < BT; r += NT) {
      *reinterpret_cast<uint4*>(W + r * LDK + DK) = z;
      *reinterpret_cast<uint4*>(qkm + r * LD64 + BT) = z;
      if (ws.KKM) *reinterpret_cast<uint4*>(ws.KKM + bh * BT * LD64 + r * LD64 + BT) = z;
    }
    for (int r = tid; r < (DV / 16) * BT; r += NT) *reinterpret_cast<uint4*>(U + r * LDU + 16) = z;
  }
}

template <class K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int DV>
cudaError_t launch_pre(const SeqMap& m, const void* q, const void* k, const void* v,
                       const void* g, const void* beta, const TcWs& ws, cudaStream_t st) {
  using bf = __nv_bfloat16;
  cudaError_t e;
  if ((e = set_smem(k_pre_tc<DV>, sizeof(PreSmem<DV>)))) return e;
  if (m.nblk_cap > 0) {
    prof_mark(st, "tc_pre");
    k_pre_tc<DV><<<dim3(m.nblk_cap, m.H), 256, sizeof(PreSmem<DV>), st>>>(
        m, (const bf*)q, (const bf*)k, (const bf*)v, (const bf*)g, (const bf*)beta, ws);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_pre(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const TcWs& ws, cudaStream_t st) {
  if (dv == 128) return launch_pre<128>(m, q, k, v, g, beta, ws, st);
  return launch_pre<256>(m, q, k, v, g, beta, ws, st);
}

}  // namespace gdn
