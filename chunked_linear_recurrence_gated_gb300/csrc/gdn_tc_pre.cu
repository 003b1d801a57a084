// Pre kernel of the bf16 tensor-core path: per 64-token block and head, the
// WY factors and masks every later step reads.
//
// Per 64-token block (StateFlow review: Pre / ST / Out with V^new, Eq. 2;
// kernel-level blocks b_{i,j}; tile size BV over the value dimension):
//   Pre : A = strictly-lower(diag(beta) K K^T * Mask), T = (I + A)^-1 (fp32),
//         W = T diag(beta Gamma) K, U = T diag(beta) V, QKM = Q K^T * Mask
//   ST  : V^new = U - W H_b ; H_{b+1} = Gamma_C H_b + K^T diag(e^{gamma_C - gamma}) V^new
//   Out : O = diag(Gamma) Q H_b + QKM V^new
// Pre also writes decay-scaled copies of the block's rows,
// K~ = diag(e^{gamma_C - gamma}) K and Q~ = diag(e^{gamma}) Q, and the per-row
// vectors (Gamma_r, e^{gamma_C - gamma_r}, gamma_r, beta_r), so that the
// sequential chains fetch every operand with one bulk copy and scale nothing
// but the state. W, K~, Q~, QKM and K K^T * Mask leave in the 128-byte-swizzled
// layout of a shared-memory tile (sw128), so a bulk copy lands them ready for
// swizzle-aware fragment loads and tensor-core descriptors.
//
// K K^T and Q K^T (64 x 64, reduced over the 128 keys) are warp-level MMAs
// and the inverse is fp32 with TF32 MMAs for its off-diagonal blocks. W and U
// are computed transposed, W^T = K^T (T diag(beta Gamma))^T and
// U^T = V^T (T diag(beta))^T, so that their 128 rows (keys, values) fill a
// tcgen05 MMA: one thread issues them from 128-byte-swizzled shared-memory
// tiles into tensor memory, the warps read the rows back into shared-memory
// tiles in the chains' layouts, and bulk copies store the tiles.
#include <cuda.h>

#include <mutex>

#include "gdn_internal.cuh"
#include "gdn_mma.cuh"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

constexpr int LDK = TC_LDK;
constexpr int LD64 = TC_LD64;
constexpr int LDU = TC_LDU;

// ------------------------------------------------------------------ Pre
// Shared memory (byte offsets from a 1024-aligned base). The swizzled K, V
// and Q tiles hold rows t with 64-wide column tiles 8192 bytes apart. Q is
// dead once Q K^T is formed: the fp32 A of the inverse takes its space (and
// 1 KB past it), then T diag(beta Gamma) and T diag(beta) (swizzled [t][j]
// tiles, the MMAs' B operands), and once the MMAs have read those, W [t][k]
// is staged there; the tile-major U is staged over K and V. At dv = 128 this
// is 72 KB, three CTAs per SM.
template <int DV>
struct PreLayout {
  static constexpr uint32_t K = 0;                 // K (swizzled)
  static constexpr uint32_t V = 16384;             // V (swizzled), DV / 64 tiles
  static constexpr uint32_t Q = V + DV * 128;      // Q (swizzled)
  static constexpr uint32_t A = Q;                 // fp32 A (fix layout); then TW, TU; then W
  static constexpr uint32_t TW = A;                // T diag(beta Gamma) [64][64] (swizzled)
  static constexpr uint32_t TU = A + 8192;         // T diag(beta) [64][64] (swizzled)
  static constexpr uint32_t TF = A + 18432;        // fp32 T (fix layout)
  static constexpr uint32_t S = TF + 18432;        // fp32 [16] rows, block-row product (fix layout)
  static constexpr uint32_t UST = 0;               // U, tile-major [DV/16][64][LDU] (u_tile_off)
  static constexpr uint32_t VEC = S + 4608;
  static constexpr uint32_t BYTES = VEC + 4 * 256 + 64;
  static constexpr uint32_t NCOL = DV == 128 ? 128 : 256;  // TMEM: W^T [0, 64), U^T [64, 64 + DV/2)
  static constexpr int CTAS = DV == 128 ? 3 : 2;          // per SM
};
static_assert(PreLayout<128>::Q % 1024 == 0 && PreLayout<256>::Q % 1024 == 0 &&
                  PreLayout<128>::TF % 1024 == 0 && PreLayout<256>::TF % 1024 == 0,
              "swizzled tiles start 1024-byte aligned");
static_assert(PreLayout<128>::Q >= (128 / 16) * BT * TC_LDU * 2 &&
                  PreLayout<256>::Q >= (256 / 16) * BT * TC_LDU * 2,
              "the tile-major U fits over K and V");
static_assert((PreLayout<128>::BYTES + 1024 + 1024) * 3 <= 228 * 1024, "three CTAs per SM at dv = 128");
static_assert((PreLayout<256>::BYTES + 1024 + 1024) * 2 <= 228 * 1024, "two CTAs per SM at dv = 256");

// Fragment loads of mma.m16n8k16 from a swizzled tile (64-wide column tiles
// `tb` bytes apart): A rows [r0, r0+16) x cols [c0, c0+16); B for two n8
// tiles from storage [n][k], rows n in [n0, n0+16), k in [k0, k0+16).
__device__ __forceinline__ void lda_sw(uint32_t* a, uint32_t base, uint32_t tb, int r0, int c0) {
  const int l = threadIdx.x & 31;
  ldsm_x4(base + sw128(r0 + (l & 7) + ((l >> 3) & 1) * 8, c0 + (l >> 4) * 8, tb), a[0], a[1], a[2],
          a[3]);
}
__device__ __forceinline__ void ldb_nk_sw(uint32_t* b, uint32_t base, uint32_t tb, int n0, int k0) {
  const int l = threadIdx.x & 31;
  const int mat = l >> 3;
  ldsm_x4(base + sw128(n0 + (l & 7) + (mat >> 1) * 8, k0 + (mat & 1) * 8, tb), b[0], b[1], b[2],
          b[3]);
}

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

// fp32 tiles of the inverse: element (r, c) at word fix(r, c), rows of 72
// words with column bit 2 flipped on rows whose bit 2 is set, so the TF32
// fragment loads of either operand role, the float2 fragment stores and the
// diagonal blocks' row stores hit 32 distinct banks.
__device__ __forceinline__ int fix(int r, int c) { return r * 72 + (c ^ (((r >> 2) & 1) << 2)); }
__device__ __forceinline__ void st2(float* base, int r, int c, float x, float y) {  // c even
  *reinterpret_cast<float2*>(base + fix(r, c)) = make_float2(x, y);
}

// T = (I + A)^-1 for strictly-lower 64 x 64 A (fp32, fix layout), NT threads.
// The four diagonal 16 x 16 blocks by fp32 forward substitution (one warp
// each); then, block row by block row (i = 1..3), warps 0..2i-1 (one n8
// column tile each) form
//   S = A[i, 0:i] T[0:i, 0:i]   and   T[i, 0:i] = -T_ii S
// with TF32 tensor-core MMAs (fp32 accumulation): the block products of
// T_ij = -T_ii sum_{m=j}^{i-1} A_im T_mj for all j < i at once.
template <int NT>
__device__ void invert_unit_lower64(const float* A, float* Tf, float* S) {
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31, g = l >> 2, t = l & 3;
  for (int idx = tid; idx < BT * 72; idx += NT) Tf[idx] = 0.f;
  __syncthreads();
  if (w < 4 && l < 16) {
    const int c = 16 * w + l;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float v = (r == l) ? 1.f : 0.f;
#pragma unroll
      for (int j = 0; j < r; ++j) v -= A[fix(16 * w + r, 16 * w + j)] * x[j];
      x[r] = v;
      Tf[fix(16 * w + r, c)] = v;
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
      // S (16 x 8, column tile nt) = A[R:R+16, 0:16i] * Tf[0:16i, 8nt:8nt+8]; fp32
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int kt = 0; kt < 2 * i; ++kt) {
        uint32_t a[4];
        a[0] = to_tf32(A[fix(R + g, 8 * kt + t)]);
        a[1] = to_tf32(A[fix(R + g + 8, 8 * kt + t)]);
        a[2] = to_tf32(A[fix(R + g, 8 * kt + t + 4)]);
        a[3] = to_tf32(A[fix(R + g + 8, 8 * kt + t + 4)]);
        const uint32_t b0 = to_tf32(Tf[fix(8 * kt + t, 8 * nt + g)]);
        const uint32_t b1 = to_tf32(Tf[fix(8 * kt + t + 4, 8 * nt + g)]);
        mma_tf32(acc, a, b0, b1);
      }
      st2(S, g, 8 * nt + 2 * t, acc[0], acc[1]);
      st2(S, g + 8, 8 * nt + 2 * t, acc[2], acc[3]);
      __syncwarp();
      // T[R:R+16, 8nt:8nt+8] = -T_ii S
      float acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kt = 0; kt < 2; ++kt) {
        uint32_t a[4];
        a[0] = to_tf32(Tf[fix(R + g, R + 8 * kt + t)]);
        a[1] = to_tf32(Tf[fix(R + g + 8, R + 8 * kt + t)]);
        a[2] = to_tf32(Tf[fix(R + g, R + 8 * kt + t + 4)]);
        a[3] = to_tf32(Tf[fix(R + g + 8, R + 8 * kt + t + 4)]);
        const uint32_t b0 = to_tf32(S[fix(8 * kt + t, 8 * nt + g)]);
        const uint32_t b1 = to_tf32(S[fix(8 * kt + t + 4, 8 * nt + g)]);
        mma_tf32(acc2, a, b0, b1);
      }
      st2(Tf, R + g, 8 * nt + 2 * t, -acc2[0], -acc2[1]);
      st2(Tf, R + g + 8, 8 * nt + 2 * t, -acc2[2], -acc2[3]);
    }
    __syncthreads();
  }
}

// 8 warps; for the warp-level products warp (rw = w & 3, cw = w >> 2) owns
// rows [16 rw, 16 rw + 16) and the cw-th half of the columns; for the
// tensor-memory read-back warp w owns lanes [32 (w & 3), +32) and the
// (w >> 2)-th half of the columns.
template <int DV>
__global__ void __launch_bounds__(256, PreLayout<DV>::CTAS)
    k_pre_tc(SeqMap m, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
             const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ g,
             const __nv_bfloat16* __restrict__ beta, TcWs ws, int seg_b0, int seg_nb,
             const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v) {
  using L = PreLayout<DV>;
  constexpr int DK = 128;
  constexpr int NT = 256;
  constexpr uint32_t TB = 8192;  // bytes between the 64-wide column tiles of K, Q, V
  BlockInfo bi;
  // the launch covers every block, or blocks [seg_b0, seg_b0 + seg_nb) of each
  // sequence (one segment of a split fixed-length forward)
  const int gb = seg_nb > 0 ? (int)(blockIdx.x / seg_nb) * m.nblk_fixed + seg_b0 + (int)(blockIdx.x % seg_nb)
                            : (int)blockIdx.x;
  const int h = blockIdx.y, H = m.H, tid = threadIdx.x;
  // Pre is the first kernel of a fixed-length call: it clears the status word,
  // which the later kernels of the call only ever set (varlen calls: the
  // block-table kernel sets it)
  if (m.cu == nullptr && gb == 0 && h == 0 && tid == 0) ws.status[0] = DEV_OK;
  if (!block_info(m, gb, bi)) return;
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sb = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
  const uint32_t su = smem_u32(sb);
  float* sA = reinterpret_cast<float*>(sb + L::A);
  float* sTf = reinterpret_cast<float*>(sb + L::TF);
  float* sS = reinterpret_cast<float*>(sb + L::S);
  float* s_g = reinterpret_cast<float*>(sb + L::VEC);
  float* s_b = s_g + BT;
  float* s_G = s_b + BT;
  float* s_dte = s_G + BT;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sb + L::VEC + 4 * 256);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sb + L::VEC + 4 * 256 + 8);
  volatile int* abort = reinterpret_cast<volatile int*>(sb + L::VEC + 4 * 256 + 16);
  uint64_t* tbar = reinterpret_cast<uint64_t*>(sb + L::VEC + 4 * 256 + 24);
  const int w = tid >> 5, l = tid & 31, gq = l >> 2, tq = l & 3;
  const int rw = w & 3, cw = w >> 2, R0 = 16 * rw;
  const int lq = w & 3, ch = w >> 2;  // TMEM lane quarter, column half
  const size_t bh = (size_t)gb * H + h;

  // K, Q, V by tensor copies (the maps view q, k, v as [B][T][H][d] with
  // 64 x 64 boxes and the 128-byte swizzle the tiles use), one thread issuing
  if (tid == 0) {
    mbar_init(tbar, 1);
    mbar_init(mbar, 1);
    *abort = 0;
    fence_mbar_init();
    mbar_arrive_expect_tx(tbar, 2 * 2 * TB + (DV / 64) * TB);
    const int tc = m.cu ? bi.tok0 : bi.lb * BT;  // token coordinate within the sequence
    const int sc = m.cu ? 0 : bi.seq;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      tma_load_4d(sb + L::K + hh * TB, &tm_k, 64 * hh, h, tc, sc, tbar);
      tma_load_4d(sb + L::Q + hh * TB, &tm_q, 64 * hh, h, tc, sc, tbar);
    }
#pragma unroll
    for (int vt = 0; vt < DV / 64; ++vt) tma_load_4d(sb + L::V + vt * TB, &tm_v, 64 * vt, h, tc, sc, tbar);
  }
  if (tid < BT) {
    const bool ok = tid < bi.len;
    const size_t off = (size_t)(bi.tok0 + tid) * H + h;
    s_g[tid] = ok ? __bfloat162float(g[off]) : 0.f;
    s_b[tid] = ok ? __bfloat162float(beta[off]) : 0.f;
  }
  if (w == 0) tmem_alloc(tslot, L::NCOL);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  block_cumsum64(s_g);
  bool ok = __all_sync(0xffffffffu, mbar_wait(tbar, 0, abort));
  // rows past the block's end: zeros (a tail of a sequence; the tensor copy
  // zero-fills only past the end of the tensor)
  if (bi.len < BT) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const int nr = BT - bi.len;
    for (int idx = tid; idx < nr * 16; idx += NT) {
      const int r = bi.len + (idx >> 4), c = (idx & 15) * 8;
      *reinterpret_cast<uint4*>(sb + L::K + sw128(r, c, TB)) = z;
      *reinterpret_cast<uint4*>(sb + L::Q + sw128(r, c, TB)) = z;
    }
    for (int idx = tid; idx < nr * (DV / 8); idx += NT) {
      const int r = bi.len + idx / (DV / 8), c = (idx % (DV / 8)) * 8;
      *reinterpret_cast<uint4*>(sb + L::V + (uint32_t)(c >> 6) * TB + sw128(r, c & 63, TB)) = z;
    }
  }
  __syncthreads();
  if (tid < BT) {
    const float gr = s_g[tid];
    const float G = __expf(gr), dte = __expf(s_g[BT - 1] - gr);
    s_G[tid] = G;
    s_dte[tid] = dte;
    float* dec = ws.dec + bh * TC_DEC_ROWS * BT;
    dec[tid] = G;
    dec[BT + tid] = dte;
    dec[2 * BT + tid] = gr;
    dec[3 * BT + tid] = s_b[tid];
  }
  __syncthreads();
  // decay-scaled copies for the chains (one bulk copy each per block),
  // K~ = diag(e^{gamma_C - gamma}) K and Q~ = diag(e^{gamma}) Q, in the
  // swizzled layout of the shared-memory tiles
  {
    unsigned char* gK = reinterpret_cast<unsigned char*>(ws.Kp + bh * BT * LDK);
    unsigned char* gQ = reinterpret_cast<unsigned char*>(ws.Qp + bh * BT * LDK);
    for (int idx = tid; idx < BT * (DK / 8); idx += NT) {
      const int r = idx / (DK / 8), c = (idx % (DK / 8)) * 8;
      const uint32_t off = sw128(r, c, TB);
      uint4 a = *reinterpret_cast<const uint4*>(sb + L::K + off);
      uint4 b = *reinterpret_cast<const uint4*>(sb + L::Q + off);
      const float sk = s_dte[r], sq = s_G[r];
      uint32_t* pa = &a.x;
      uint32_t* pb = &b.x;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = unpack_bf16(pa[e]), y = unpack_bf16(pb[e]);
        pa[e] = pack_bf16(sk * x.x, sk * x.y);
        pb[e] = pack_bf16(sq * y.x, sq * y.y);
      }
      *reinterpret_cast<uint4*>(gK + off) = a;
      *reinterpret_cast<uint4*>(gQ + off) = b;
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
      lda_sw(ak, su + L::K, TB, R0, 16 * kc);
      lda_sw(aq, su + L::Q, TB, R0, 16 * kc);
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        uint32_t b[4];
        ldb_nk_sw(b, su + L::K, TB, 32 * cw + 16 * jj, 16 * kc);
        mma16816(kk[2 * jj], ak, b[0], b[1]);
        mma16816(kk[2 * jj + 1], ak, b[2], b[3]);
        mma16816(qk[2 * jj], aq, b[0], b[1]);
        mma16816(qk[2 * jj + 1], aq, b[2], b[3]);
      }
    }
    __nv_bfloat16* qkm = ws.QKM + bh * BT * LD64;
    __syncthreads();  // every warp is done reading Q before A overwrites it
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = R0 + gq + 8 * hf;
        const int c = 32 * cw + 8 * j + 2 * tq;
        const float gr = s_g[r];
        const float d0 = (c <= r) ? __expf(gr - s_g[c]) : 0.f;
        const float d1 = (c + 1 <= r) ? __expf(gr - s_g[c + 1]) : 0.f;
        const float br = s_b[r];
        const float km0 = (c < r) ? kk[j][2 * hf] * d0 : 0.f;
        const float km1 = (c + 1 < r) ? kk[j][2 * hf + 1] * d1 : 0.f;
        st2(sA, r, c, br * km0, br * km1);
        if (ws.KKM)
          *reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(ws.KKM + bh * BT * LD64) +
                                       sw128(r, c, 0)) = pack_bf16(km0, km1);
        *reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(qkm) + sw128(r, c, 0)) =
            pack_bf16(qk[j][2 * hf] * d0, qk[j][2 * hf + 1] * d1);
      }
  }
  __syncthreads();
  invert_unit_lower64<NT>(sA, sTf, sS);
  // Tw = T diag(beta Gamma), Tu = T diag(beta) as swizzled [t][j] tiles; T itself for the backward
  for (int idx = 2 * tid; idx < BT * BT; idx += 2 * NT) {  // column pairs
    const int r = idx >> 6, c = idx & 63;
    const float2 t = *reinterpret_cast<const float2*>(&sTf[fix(r, c)]);
    const float2 bc = *reinterpret_cast<const float2*>(&s_b[c]);
    const float2 Gc = *reinterpret_cast<const float2*>(&s_G[c]);
    *reinterpret_cast<uint32_t*>(sb + L::TW + sw128(r, c, 0)) =
        pack_bf16(t.x * bc.x * Gc.x, t.y * bc.y * Gc.y);
    *reinterpret_cast<uint32_t*>(sb + L::TU + sw128(r, c, 0)) = pack_bf16(t.x * bc.x, t.y * bc.y);
    if (ws.T) *reinterpret_cast<uint32_t*>(ws.T + bh * BT * BT + idx) = pack_bf16(t.x, t.y);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();

  // W^T = K^T Tw^T -> TMEM columns [0, 64); U^T = V^T Tu^T -> [64, 64 + 64 DV/128)
  if (tid == 0) {
    tc_fence_after();
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      umma_bf16(tmem, umma_desc(su + L::K + 2048 * s, TB, 1024),
                umma_desc(su + L::TW + 32 * s, 16, 1024), umma_idesc(128, 64, 1, 0), s > 0);
      const uint64_t bu = umma_desc(su + L::TU + 32 * s, 16, 1024);
#pragma unroll
      for (int mh = 0; mh < DV / 128; ++mh)
        umma_bf16(tmem + 64 + 64 * mh, umma_desc(su + L::V + 2 * TB * mh + 2048 * s, TB, 1024), bu,
                  umma_idesc(128, 64, 1, 0), s > 0);
    }
    umma_commit(mbar);
  }
  ok = __all_sync(0xffffffffu, mbar_wait(mbar, 0, abort)) && ok;  // warp-uniform for tcgen05.ld
  tc_fence_after();
  // read back: lane = key k (W^T) or value v (U^T), 32 tokens per warp; staged as
  // W [t][k] (swizzled 64-key tiles) in A's space and U tile-major at the start
  if (ok) {
    const uint32_t lane_base = tmem + ((uint32_t)(32 * lq) << 16);
    unsigned char* Wst = sb + L::A;
    __nv_bfloat16* Ust = reinterpret_cast<__nv_bfloat16*>(sb + L::UST);
#pragma unroll
    for (int part = 0; part <= DV / 128; ++part) {
      float vv[32];
      tmem_ld16(lane_base + 64 * part + 32 * ch, vv);
      tmem_ld16(lane_base + 64 * part + 32 * ch + 16, vv + 16);
      if (part == 0) {
        const int kk = 32 * lq + l;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          *reinterpret_cast<__nv_bfloat16*>(Wst + sw128(32 * ch + i, kk, TB)) = __float2bfloat16_rn(vv[i]);
      } else {
        const int vv_ = 128 * (part - 1) + 32 * lq + l;
        __nv_bfloat16* tile = Ust + (size_t)(vv_ >> 4) * BT * LDU;
        // lanes 16-31 fill the next 16-value tile, whose rows sit on the same
        // banks: they take the tokens in swapped pairs, so each store is one wavefront
        const bool hi = l >= 16;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          tile[u_tile_off(32 * ch + (hi ? (i ^ 1) : i), vv_ & 15)] = __float2bfloat16_rn(hi ? vv[i ^ 1] : vv[i]);
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    if (ok) {
      bulk_s2g(ws.W + bh * BT * LDK, sb + L::A, BT * DK * 2);
      bulk_s2g(ws.U + bh * (DV / 16) * BT * LDU, sb + L::UST, (DV / 16) * BT * LDU * 2);
      bulk_commit();
    } else {
      ws.status[0] = DEV_TIMEOUT;
    }
  }
  if (tid == 0) bulk_wait_read();  // the staged tiles stay valid until read
  __syncthreads();
  if (w == 0) tmem_dealloc(tmem, L::NCOL);
}

template <class K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  });
  return fn;
}

}  // namespace

// View of a [B][T][H][d] bf16 tensor (varlen: [1][total][H][d]) as a 4-D map
// with 64-element x 1 head x 64-token boxes and the 128-byte swizzle.
cudaError_t make_tok_map(CUtensorMap* map, const void* base, int d, const SeqMap& m) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const bool varlen = m.cu != nullptr;
  const cuuint64_t T = varlen ? (cuuint64_t)m.T_total : (cuuint64_t)m.T_fixed;
  const cuuint64_t Bn = varlen ? 1 : (cuuint64_t)m.nseq;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)m.H, T, Bn};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)m.H * d * 2,
                                 (cuuint64_t)m.H * d * 2 * T};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)BT, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}


// View of a per-block-head workspace array [nbh][rows][row_stride] (bf16) as a
// 3-D map whose boxes are 64 elements x box_rows rows of one block-head, with
// the 128-byte swizzle.
cudaError_t make_ws_map(CUtensorMap* map, const void* base, int inner, int rows, int row_stride,
                        long long nbh, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)nbh};
  const cuuint64_t strides[2] = {(cuuint64_t)row_stride * 2, (cuuint64_t)row_stride * 2 * rows};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

template <int DV>
cudaError_t launch_pre(const SeqMap& m, const void* q, const void* k, const void* v,
                       const void* g, const void* beta, const TcWs& ws, int b0, int nb,
                       cudaStream_t st, bool mark) {
  using bf = __nv_bfloat16;
  cudaError_t e;
  constexpr size_t smem = PreLayout<DV>::BYTES + 1024;  // + alignment of the base
  if ((e = set_smem(k_pre_tc<DV>, smem))) return e;
  const int gx = nb > 0 ? nb * m.nseq : m.nblk_cap;
  if (gx > 0) {
    alignas(64) CUtensorMap tq, tk, tv;
    if ((e = make_tok_map(&tq, q, 128, m)) || (e = make_tok_map(&tk, k, 128, m)) ||
        (e = make_tok_map(&tv, v, DV, m)))
      return e;
    if (mark) prof_mark(st, "tc_pre");
    k_pre_tc<DV><<<dim3(gx, m.H), 256, smem, st>>>(m, (const bf*)q, (const bf*)k, (const bf*)v,
                                                 (const bf*)g, (const bf*)beta, ws, b0, nb, tq, tk,
                                                 tv);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc_pre(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const TcWs& ws, int b0, int nb,
                   cudaStream_t st, bool mark) {
  if (dv == 128) return launch_pre<128>(m, q, k, v, g, beta, ws, b0, nb, st, mark);
  return launch_pre<256>(m, q, k, v, g, beta, ws, b0, nb, st, mark);
}

}  // namespace gdn
