// C-ABI entry points (include/gdn.h): argument checks, workspace carving,
// varlen block tables, and dispatch to the kernel families.
#include <stdint.h>

#include "../../include/gdn.h"
#include "../../include/gdn_profile.h"
#include "gdn_internal.cuh"
#include "gdn_mma.cuh"

namespace gdn {

// ------------------------------------------------------------ timing hook
namespace {
cudaEvent_t* g_prof_ev = nullptr;
int g_prof_cap = 0;
int g_prof_n = 0;
const char* g_prof_names[4096];
}  // namespace

void prof_mark(cudaStream_t st, const char* next) {
  if (!g_prof_ev || g_prof_n >= g_prof_cap) return;
  if (cudaEventRecord(g_prof_ev[g_prof_n], st) != cudaSuccess) return;
  g_prof_names[g_prof_n] = next;
  ++g_prof_n;
}

// ------------------------------------------------------------ varlen block tables
// One CTA: validates cu_seqlens (cu[0] = 0, non-decreasing, cu[nseq] = T),
// numbers the 64-token blocks of every sequence (each sequence's grid starts
// at its first token) and records the owning sequence of each block. A
// malformed array sets the status word and leaves every table empty, so no
// kernel does any work. order (blk0 + nseq + 1) lists the sequences longest
// first (ties by index; index order past 4096 sequences): the sequential
// chains start their CTAs in that order, so the longest chains do not trail.
__global__ void k_varlen_prep(const int* __restrict__ cu, int nseq, int T, int nblk_cap,
                              int* blk0, int* blk_seq, int* status) {
  __shared__ int bad;
  if (threadIdx.x == 0) bad = (cu[0] != 0 || cu[nseq] != T) ? 1 : 0;
  __syncthreads();
  for (int s = threadIdx.x; s < nseq; s += blockDim.x)
    if (cu[s + 1] < cu[s]) bad = 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int s = 0; s < nseq; ++s) {
      blk0[s] = acc;
      if (!bad) acc += (cu[s + 1] - cu[s] + BT - 1) / BT;
    }
    blk0[nseq] = acc;
    if (acc > nblk_cap) bad = 1;  // cannot happen for a valid array
    status[0] = bad ? DEV_BAD_CU_SEQLENS : DEV_OK;
  }
  __syncthreads();
  if (bad) {
    for (int gb = threadIdx.x; gb < nblk_cap; gb += blockDim.x) blk_seq[gb] = -1;
    for (int s = threadIdx.x; s <= nseq; s += blockDim.x) blk0[s] = 0;
    for (int s = threadIdx.x; s < nseq; s += blockDim.x) blk0[nseq + 1 + s] = s;
    return;
  }
  for (int s = threadIdx.x; s < nseq; s += blockDim.x)
    for (int gb = blk0[s]; gb < blk0[s + 1]; ++gb) blk_seq[gb] = s;
  for (int gb = blk0[nseq] + threadIdx.x; gb < nblk_cap; gb += blockDim.x) blk_seq[gb] = -1;
  int* order = blk0 + nseq + 1;
  for (int s = threadIdx.x; s < nseq; s += blockDim.x) {
    int rank = s;
    if (nseq <= 4096) {
      const int n = blk0[s + 1] - blk0[s];
      rank = 0;
      for (int o = 0; o < nseq; ++o) {
        const int no = blk0[o + 1] - blk0[o];
        rank += (no > n || (no == n && o < s)) ? 1 : 0;
      }
    }
    order[rank] = s;
  }
}

cudaError_t varlen_prep(const int* cu, int nseq, int T, int nblk_cap, int* blk0, int* blk_seq,
                        int* status, cudaStream_t st) {
  prof_mark(st, "varlen_prep");
  k_varlen_prep<<<1, 1024, 0, st>>>(cu, nseq, T, nblk_cap, blk0, blk_seq, status);
  return cudaGetLastError();
}

__global__ void k_status_ok(int* status) { status[0] = DEV_OK; }

cudaError_t reset_status(int* status, cudaStream_t st) {
  prof_mark(st, "status");
  k_status_ok<<<1, 1, 0, st>>>(status);
  return cudaGetLastError();
}

// Failure-detection self-check: one bounded wait on an mbarrier that never
// completes (its one expected arrival never comes).
__global__ void k_diag_wait(int* status, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = mbar_wait(&bar, 0, &abort, limit);
  __syncthreads();
  if (threadIdx.x == 0) status[0] = ok ? DEV_OK : DEV_TIMEOUT;
}

}  // namespace gdn

namespace {

using namespace gdn;

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

struct Plan {
  int B, T, H, dk, dv, dtype;
  int nseq;       // sequences (B for fixed-length calls)
  int nblk_cap;   // global 64-token blocks launched
  bool varlen;
};

bool supported(const gdn_shape* s) {
  return (s->dtype == GDN_DTYPE_F32 || s->dtype == GDN_DTYPE_BF16) &&
         (s->dk == 64 || s->dk == 128) && (s->dv == 64 || s->dv == 128 || s->dv == 256);
}

gdn_status plan_shape(const gdn_shape* s, bool varlen, int nseq, Plan* p) {
  if (!s) return GDN_ERR_INVALID_ARG;
  if (s->B < 1 || s->T < 0 || s->H < 1 || s->H > 65535 || s->dk < 1 || s->dv < 1)
    return GDN_ERR_INVALID_ARG;
  if (!supported(s)) return GDN_ERR_UNSUPPORTED;
  p->B = s->B; p->T = s->T; p->H = s->H; p->dk = s->dk; p->dv = s->dv; p->dtype = s->dtype;
  p->varlen = varlen;
  const long long nbs = ((long long)s->T + BT - 1) / BT;
  long long nblk;
  if (varlen) {
    if (s->B != 1 || nseq < 1) return GDN_ERR_INVALID_ARG;
    p->nseq = nseq;
    nblk = nbs + nseq;
  } else {
    p->nseq = s->B;
    nblk = nbs * s->B;
  }
  if (nblk > (1ll << 30) || (long long)p->nseq * p->H * (p->dv / 16) > (1ll << 30) ||
      (long long)s->B * s->T > (1ll << 31) - 1)
    return GDN_ERR_INVALID_ARG;
  p->nblk_cap = (int)nblk;
  return GDN_OK;
}

// Kernel family for a shape: 2 = bf16 tensor-core kernels, 1 = fp32-arithmetic
// SIMT kernels. Depends only on dtype, dk and dv (never on T), so chunked and
// unchunked calls of one problem always run the same arithmetic.
int path_of(const Plan& p) {
  if (p.dtype == GDN_DTYPE_BF16 && p.dk == 128 && (p.dv == 128 || p.dv == 256)) return 2;
  return 1;
}

struct Carve {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off = up(off + bytes);
    return o;
  }
};

// Workspace layout of the SIMT kernels. The first 256 bytes hold the status word.
size_t simt_layout(const Plan& p, bool bwd, SimtWs* ws, int** blk0, int** blk_seq, char* base) {
  Carve c;
  const size_t nbh = (size_t)p.nblk_cap * p.H;
  const size_t o_status = c.take(kAlign);
  // blk0 [nseq + 1], then the sequences in the order the chains take them [nseq]
  const size_t o_blk0 = p.varlen ? c.take(sizeof(int) * (2 * (size_t)p.nseq + 1)) : 0;
  const size_t o_blks = p.varlen ? c.take(sizeof(int) * (size_t)p.nblk_cap) : 0;
  const size_t o_gam = c.take(4 * nbh * BT);
  const size_t o_W = c.take(4 * nbh * BT * p.dk);
  const size_t o_U = c.take(4 * nbh * BT * p.dv);
  const size_t o_Hb = c.take(4 * nbh * p.dk * p.dv);
  const size_t o_Vn = c.take(4 * nbh * BT * p.dv);
  size_t o_T = 0, o_dH = 0, o_dVn = 0;
  if (bwd) {
    o_T = c.take(4 * nbh * BT * BT);
    o_dH = c.take(4 * nbh * p.dk * p.dv);
    o_dVn = c.take(4 * nbh * BT * p.dv);
  }
  if (base) {
    ws->status = (int*)(base + o_status);
    ws->gam = (float*)(base + o_gam);
    ws->W = (float*)(base + o_W);
    ws->U = (float*)(base + o_U);
    ws->Hb = (float*)(base + o_Hb);
    ws->Vn = (float*)(base + o_Vn);
    ws->Tm = bwd ? (float*)(base + o_T) : nullptr;
    ws->dH = bwd ? (float*)(base + o_dH) : nullptr;
    ws->dVn = bwd ? (float*)(base + o_dVn) : nullptr;
    *blk0 = p.varlen ? (int*)(base + o_blk0) : nullptr;
    *blk_seq = p.varlen ? (int*)(base + o_blks) : nullptr;
  }
  return c.off;
}

// Workspace layout of the tensor-core kernels (bf16 intermediates).
// Per-block products of the Pre kernel (dec, W, U, QKM, Kp, Qp; the backward
// also T and KKM), carved from `base` (nullptr: sizes only) starting at offset 0.
void carve_pre(const Plan& p, bool bwd, Carve& c, TcWs* ws, char* base) {
  using bf = __nv_bfloat16;
  const size_t nbh = (size_t)p.nblk_cap * p.H;
  const size_t o_dec = c.take(4 * nbh * TC_DEC_ROWS * BT);
  const size_t o_W = c.take(2 * nbh * BT * TC_LDK);
  const size_t o_U = c.take(2 * nbh * (p.dv / 16) * BT * TC_LDU);
  const size_t o_QKM = c.take(2 * nbh * BT * TC_LD64);
  const size_t o_Kp = c.take(2 * nbh * BT * TC_LDK);
  const size_t o_Qp = c.take(2 * nbh * BT * TC_LDK);
  const size_t o_T = bwd ? c.take(2 * nbh * BT * BT) : 0;
  const size_t o_KKM = bwd ? c.take(2 * nbh * BT * TC_LD64) : 0;
  if (base) {
    ws->dec = (float*)(base + o_dec);
    ws->W = (bf*)(base + o_W);
    ws->U = (bf*)(base + o_U);
    ws->QKM = (bf*)(base + o_QKM);
    ws->Kp = (bf*)(base + o_Kp);
    ws->Qp = (bf*)(base + o_Qp);
    ws->T = bwd ? (bf*)(base + o_T) : nullptr;
    ws->KKM = bwd ? (bf*)(base + o_KKM) : nullptr;
  }
}

// Bytes of the saved forward products (gdn_chunk_fwd_save / gdn_chunk_bwd_saved):
// the Pre products with T and K K^T, and the chain's H_b and V^new per block.
size_t saved_layout(const Plan& p, TcWs* ws, char* base) {
  Carve c;
  carve_pre(p, true, c, ws, base);
  const size_t nbh = (size_t)p.nblk_cap * p.H;
  const size_t o_Hb = c.take(2 * nbh * p.dv * p.dk);
  const size_t o_Vn = c.take(2 * nbh * p.dv * BT);
  if (base) {
    ws->HbT = (__nv_bfloat16*)(base + o_Hb);
    ws->VnT = (__nv_bfloat16*)(base + o_Vn);
  }
  return c.off;
}

// Workspace layout of the tensor-core kernels. The first 256 bytes hold the
// status word. WS_FWD / WS_BWD hold the Pre products themselves (WS_BWD also
// H_b and V^new); WS_SAVED leaves those to a separate saved-products buffer.
enum WsKind { WS_FWD = 0, WS_BWD = 1, WS_SAVED = 2 };
size_t tc_layout(const Plan& p, int kind, TcWs* ws, int** blk0, int** blk_seq, char* base) {
  Carve c;
  const bool bwd = kind != WS_FWD;
  const size_t nbh = (size_t)p.nblk_cap * p.H;
  const size_t o_status = c.take(kAlign);
  // blk0 [nseq + 1], then the sequences in the order the chains take them [nseq]
  const size_t o_blk0 = p.varlen ? c.take(sizeof(int) * (2 * (size_t)p.nseq + 1)) : 0;
  const size_t o_blks = p.varlen ? c.take(sizeof(int) * (size_t)p.nblk_cap) : 0;
  if (kind != WS_SAVED) {
    Carve pc;
    carve_pre(p, bwd, pc, ws, nullptr);
    const size_t o_pre = c.take(pc.off);
    if (base) {
      Carve pb;
      carve_pre(p, bwd, pb, ws, base + o_pre);
    }
  }
  const bool states = kind == WS_BWD;  // WS_SAVED: H_b, V^new live with the saved products
  // fp32 state between the segments of a split forward (forward workspaces)
  const size_t sbytes = 4 * (size_t)p.nseq * p.H * p.dk * p.dv;
  const size_t o_S0 = kind != WS_BWD ? c.take(sbytes) : 0;
  const size_t o_S1 = kind != WS_BWD ? c.take(sbytes) : 0;
  size_t o_Hb = 0, o_Vn = 0, o_dH = 0, o_dVn = 0;
  if (states) {
    o_Hb = c.take(2 * nbh * p.dv * p.dk);
    o_Vn = c.take(2 * nbh * p.dv * BT);
  }
  if (bwd) {
    o_dH = c.take(2 * nbh * p.dv * p.dk);
    o_dVn = c.take(2 * nbh * p.dv * BT);
  }
  if (base) {
    using bf = __nv_bfloat16;
    ws->status = (int*)(base + o_status);
    ws->HbT = states ? (bf*)(base + o_Hb) : nullptr;
    ws->VnT = states ? (bf*)(base + o_Vn) : nullptr;
    ws->dHT = bwd ? (bf*)(base + o_dH) : nullptr;
    ws->dVnT = bwd ? (bf*)(base + o_dVn) : nullptr;
    ws->Sseg[0] = kind != WS_BWD ? (float*)(base + o_S0) : nullptr;
    ws->Sseg[1] = kind != WS_BWD ? (float*)(base + o_S1) : nullptr;
    *blk0 = p.varlen ? (int*)(base + o_blk0) : nullptr;
    *blk_seq = p.varlen ? (int*)(base + o_blks) : nullptr;
  }
  return c.off;
}

size_t ws_bytes(const Plan& p, int kind) {
  int *a, *b;
  if (path_of(p) == 2) {
    TcWs w;
    return tc_layout(p, kind, &w, &a, &b, nullptr);
  }
  SimtWs w;
  return simt_layout(p, kind != WS_FWD, &w, &a, &b, nullptr);
}

size_t saved_bytes(const Plan& p) {
  if (path_of(p) == 2) {
    TcWs w;
    return saved_layout(p, &w, nullptr);
  }
  return kAlign;  // the fp32 SIMT kernels keep nothing between the two calls
}

bool al(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

// Tensor arguments: [.., d] tensors need 16-byte alignment, [B, T, H] tensors
// element alignment; states 16 bytes. Returns false on a violation.
bool check_tensor(const void* p, bool required, size_t align) {
  if (!p) return !required;
  return al(p, align);
}

SeqMap make_map(const Plan& p, const int* cu, const int* blk0, const int* blk_seq) {
  SeqMap m;
  m.cu = p.varlen ? cu : nullptr;
  m.blk0 = blk0;
  m.blk_seq = blk_seq;
  m.order = p.varlen ? blk0 + p.nseq + 1 : nullptr;
  m.nseq = p.nseq;
  m.T_fixed = p.varlen ? 0 : p.T;
  m.nblk_fixed = p.varlen ? 0 : (p.T + BT - 1) / BT;
  m.nblk_cap = p.nblk_cap;
  m.H = p.H;
  m.T_total = (long long)p.B * p.T;
  return m;
}

// Split of a fixed-length tensor-core forward (state-transition / dense-kernel
// overlap). The default is the setting measured fastest on the benchmark's
// 32768-token chunks: no split (a chain CTA holds ~205 KB of shared memory, so
// Pre cannot share its SMs, and a chain carrying 32 value columns per CTA to
// leave SMs free runs 1.6x slower per step than the overlap gains);
// gdn_diag_set_fwd_split overrides it for measurements.
int g_split_nseg = 0;       // 0: default policy
int g_split_permille = 0;   // first segment's share of the blocks when nseg = 2 (0: equal)
int g_split_rg = 0;         // chain value-row groups (0: default)
constexpr int kDefaultSegments = 1;
constexpr int kDefaultSplitRG = 2;

FwdSplit fwd_split(const Plan& p, bool allow) {
  FwdSplit sp;
  const int nblk = (p.T + BT - 1) / BT;
  int nseg = g_split_nseg > 0 ? g_split_nseg : kDefaultSegments;
  if (!allow || p.varlen) nseg = 1;
  nseg = nseg < 1 ? 1 : (nseg > FwdSplit::kMaxSeg ? FwdSplit::kMaxSeg : nseg);
  if (nseg > nblk) nseg = nblk > 0 ? nblk : 1;
  sp.nseg = nseg;
  sp.chain_rg = g_split_rg > 0 ? g_split_rg : (nseg > 1 ? kDefaultSplitRG : 1);
  if (g_split_rg <= 0 && nseg == 1) {
    // A chain CTA per 16 value columns of each (sequence, head) is fastest while
    // they fit the GPU in one wave; beyond that 32 columns per CTA do the same
    // work in fewer CTA-steps (a step with 32 columns costs ~1.5x one with 16).
    // The columns' arithmetic is the same either way, bit for bit.
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0 &&
        (long long)p.nseq * p.H * (p.dv / 16) > sms)
      sp.chain_rg = 2;
  }
  sp.b[0] = 0;
  for (int i = 1; i < nseg; ++i) sp.b[i] = (int)(((long long)nblk * i) / nseg);
  if (nseg == 2 && g_split_permille > 0) {
    int b1 = (int)(((long long)nblk * g_split_permille + 500) / 1000);
    sp.b[1] = b1 < 1 ? 1 : (b1 > nblk - 1 ? nblk - 1 : b1);
  }
  sp.b[nseg] = nblk;
  return sp;
}

// `saved` (nullable): the forward also keeps its Pre products there, with the
// backward's T and K K^T tiles, for run_bwd to read instead of recomputing.
gdn_status run_fwd(const Plan& p, const int* cu, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const float* S_in, void* o, float* S_out,
                   void* saved, size_t savedb, void* ws, size_t wsb, void* stream,
                   bool allow_split = true) {
  const size_t esz = p.dtype == GDN_DTYPE_F32 ? 4 : 2;
  const bool any = p.T > 0;
  if (!check_tensor(q, any, 16) || !check_tensor(k, any, 16) || !check_tensor(v, any, 16) ||
      !check_tensor(g, any, esz) || !check_tensor(beta, any, esz) || !check_tensor(o, any, 16) ||
      !check_tensor(S_in, false, 16) || !check_tensor(S_out, false, 16))
    return GDN_ERR_INVALID_ARG;
  if (p.varlen && (!cu || !al(cu, 4))) return GDN_ERR_INVALID_ARG;
  const int kind = saved ? WS_SAVED : WS_FWD;
  if (!ws || !al(ws, kAlign) || wsb < ws_bytes(p, kind)) return GDN_ERR_WORKSPACE;
  if (saved && (!al(saved, kAlign) || savedb < saved_bytes(p))) return GDN_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  int *blk0, *blk_seq;
  cudaError_t e;
  if (path_of(p) == 2) {
    TcWs w;
    tc_layout(p, kind, &w, &blk0, &blk_seq, (char*)ws);
    if (saved) {
      saved_layout(p, &w, (char*)saved);  // the forward chain then also keeps H_b, V^new
      w.dHT = w.dVnT = nullptr;
    }
    if (p.varlen && (e = varlen_prep(cu, p.nseq, p.T, p.nblk_cap, blk0, blk_seq, w.status, st)))
      return GDN_ERR_CUDA;
    // the status word is cleared by the call's first kernel (the block-table
    // kernel of a varlen call, else Pre); a call with no block runs no Pre
    if (!p.varlen && p.nblk_cap == 0 && (e = reset_status(w.status, st))) return GDN_ERR_CUDA;
    const SeqMap m = make_map(p, cu, blk0, blk_seq);
    e = tc_fwd(m, p.dv, q, k, v, g, beta, S_in, o, S_out, w, fwd_split(p, allow_split), st);
    return e ? GDN_ERR_CUDA : GDN_OK;
  }
  SimtWs w;
  simt_layout(p, false, &w, &blk0, &blk_seq, (char*)ws);
  (void)savedb;
  if (p.varlen)
    e = varlen_prep(cu, p.nseq, p.T, p.nblk_cap, blk0, blk_seq, w.status, st);
  else {
    e = reset_status(w.status, st);
  }
  if (e) return GDN_ERR_CUDA;
  const SeqMap m = make_map(p, cu, blk0, blk_seq);
  e = simt_fwd(m, p.dk, p.dv, p.dtype, q, k, v, g, beta, S_in, o, S_out, w, st);
  return e ? GDN_ERR_CUDA : GDN_OK;
}

// `saved` (nullable): Pre products written by run_fwd on the same inputs; the
// Pre kernel is then not launched again.
gdn_status run_bwd(const Plan& p, const int* cu, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const float* S_in, const void* dout,
                   const float* dS_out, void* dq, void* dk, void* dv, void* dg, void* dbeta,
                   float* dS_in, const void* saved, size_t savedb, void* ws, size_t wsb,
                   void* stream) {
  const size_t esz = p.dtype == GDN_DTYPE_F32 ? 4 : 2;
  const bool any = p.T > 0;
  if (!check_tensor(q, any, 16) || !check_tensor(k, any, 16) || !check_tensor(v, any, 16) ||
      !check_tensor(g, any, esz) || !check_tensor(beta, any, esz) ||
      !check_tensor(dout, any, 16) || !check_tensor(dq, any, 16) ||
      !check_tensor(dk, any, 16) || !check_tensor(dv, any, 16) || !check_tensor(dg, any, esz) ||
      !check_tensor(dbeta, any, esz) || !check_tensor(S_in, false, 16) ||
      !check_tensor(dS_out, false, 16) || !check_tensor(dS_in, false, 16))
    return GDN_ERR_INVALID_ARG;
  if (p.varlen && (!cu || !al(cu, 4))) return GDN_ERR_INVALID_ARG;
  const int kind = saved ? WS_SAVED : WS_BWD;
  if (!ws || !al(ws, kAlign) || wsb < ws_bytes(p, kind)) return GDN_ERR_WORKSPACE;
  if (saved && (!al(saved, kAlign) || savedb < saved_bytes(p))) return GDN_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  int *blk0, *blk_seq;
  cudaError_t e;
  if (path_of(p) == 2) {
    TcWs w;
    tc_layout(p, kind, &w, &blk0, &blk_seq, (char*)ws);
    if (saved) saved_layout(p, &w, (char*)saved);
    if (p.varlen && (e = varlen_prep(cu, p.nseq, p.T, p.nblk_cap, blk0, blk_seq, w.status, st)))
      return GDN_ERR_CUDA;
    // Pre clears the status word when it runs; the backward from kept
    // products (or a call with no block) starts with the reverse chain instead
    if (!p.varlen && (saved || p.nblk_cap == 0) && (e = reset_status(w.status, st)))
      return GDN_ERR_CUDA;
    const SeqMap m = make_map(p, cu, blk0, blk_seq);
    e = tc_bwd(m, p.dv, q, k, v, g, beta, S_in, dout, dS_out, dq, dk, dv, dg, dbeta, dS_in, w,
               saved == nullptr, st);
    return e ? GDN_ERR_CUDA : GDN_OK;
  }
  SimtWs w;
  simt_layout(p, true, &w, &blk0, &blk_seq, (char*)ws);
  if (p.varlen)
    e = varlen_prep(cu, p.nseq, p.T, p.nblk_cap, blk0, blk_seq, w.status, st);
  else {
    e = reset_status(w.status, st);
  }
  if (e) return GDN_ERR_CUDA;
  const SeqMap m = make_map(p, cu, blk0, blk_seq);
  e = simt_bwd(m, p.dk, p.dv, p.dtype, q, k, v, g, beta, S_in, dout, dS_out, dq, dk, dv, dg,
               dbeta, dS_in, w, st);
  return e ? GDN_ERR_CUDA : GDN_OK;
}

}  // namespace

namespace gdn {
// gdn_chunk_fwd without the split forward (which creates internal streams on
// first use): the no-allocation entry point's forward.
gdn_status chunk_fwd_unsplit(const gdn_shape* shape, const void* q, const void* k, const void* v,
                             const void* g, const void* beta, const float* S_in, void* o,
                             float* S_out, void* workspace, size_t workspace_bytes, void* stream) {
  Plan p;
  gdn_status s = plan_shape(shape, false, 0, &p);
  if (s != GDN_OK) return s;
  return run_fwd(p, nullptr, q, k, v, g, beta, S_in, o, S_out, nullptr, 0, workspace,
                 workspace_bytes, stream, false);
}
}  // namespace gdn

extern "C" {

void gdn_diag_set_fwd_split(int segments, int first_permille, int chain_rg) {
  g_split_nseg = segments > 0 ? segments : 0;
  g_split_permille = first_permille > 0 && first_permille < 1000 ? first_permille : 0;
  g_split_rg = chain_rg == 1 || chain_rg == 2 ? chain_rg : 0;
}

size_t gdn_chunk_workspace_bytes(const gdn_shape* shape, int is_bwd) {
  Plan p;
  if (plan_shape(shape, false, 0, &p) != GDN_OK) return 0;
  if (is_bwd != GDN_WS_SAVED) is_bwd = is_bwd != 0 ? WS_BWD : WS_FWD;
  return ws_bytes(p, is_bwd);
}

size_t gdn_varlen_workspace_bytes(const gdn_shape* shape, int nseq, int is_bwd) {
  Plan p;
  if (plan_shape(shape, true, nseq, &p) != GDN_OK) return 0;
  return ws_bytes(p, is_bwd != 0 ? WS_BWD : WS_FWD);
}

gdn_status gdn_chunk_fwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, const float* S_in, void* o,
                         float* S_out, void* workspace, size_t workspace_bytes, void* stream) {
  Plan p;
  gdn_status s = plan_shape(shape, false, 0, &p);
  if (s != GDN_OK) return s;
  return run_fwd(p, nullptr, q, k, v, g, beta, S_in, o, S_out, nullptr, 0, workspace,
                 workspace_bytes, stream);
}

size_t gdn_chunk_saved_bytes(const gdn_shape* shape) {
  Plan p;
  if (plan_shape(shape, false, 0, &p) != GDN_OK) return 0;
  return saved_bytes(p);
}

gdn_status gdn_chunk_fwd_save(const gdn_shape* shape, const void* q, const void* k,
                              const void* v, const void* g, const void* beta, const float* S_in,
                              void* o, float* S_out, void* saved, size_t saved_bytes_,
                              void* workspace, size_t workspace_bytes, void* stream) {
  Plan p;
  gdn_status s = plan_shape(shape, false, 0, &p);
  if (s != GDN_OK) return s;
  if (!saved) return GDN_ERR_WORKSPACE;
  return run_fwd(p, nullptr, q, k, v, g, beta, S_in, o, S_out, saved, saved_bytes_, workspace,
                 workspace_bytes, stream);
}

gdn_status gdn_chunk_bwd_saved(const gdn_shape* shape, const void* q, const void* k,
                               const void* v, const void* g, const void* beta,
                               const float* S_in, const void* dout, const float* dS_out,
                               void* dq, void* dk, void* dv, void* dg, void* dbeta, float* dS_in,
                               const void* saved, size_t saved_bytes_, void* workspace,
                               size_t workspace_bytes, void* stream) {
  Plan p;
  gdn_status s = plan_shape(shape, false, 0, &p);
  if (s != GDN_OK) return s;
  if (!saved) return GDN_ERR_WORKSPACE;
  return run_bwd(p, nullptr, q, k, v, g, beta, S_in, dout, dS_out, dq, dk, dv, dg, dbeta, dS_in,
                 saved, saved_bytes_, workspace, workspace_bytes, stream);
}

gdn_status gdn_chunk_bwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, const float* S_in, const void* dout,
                         const float* dS_out, void* dq, void* dk, void* dv, void* dg,
                         void* dbeta, float* dS_in, void* workspace, size_t workspace_bytes,
                         void* stream) {
  Plan p;
  gdn_status s = plan_shape(shape, false, 0, &p);
  if (s != GDN_OK) return s;
  return run_bwd(p, nullptr, q, k, v, g, beta, S_in, dout, dS_out, dq, dk, dv, dg, dbeta, dS_in,
                 nullptr, 0, workspace, workspace_bytes, stream);
}

gdn_status gdn_varlen_fwd(const gdn_shape* shape, const int* cu_seqlens, int nseq,
                          const void* q, const void* k, const void* v, const void* g,
                          const void* beta, const float* S0, void* o, float* S_final,
                          void* workspace, size_t workspace_bytes, void* stream) {
  Plan p;
  gdn_status s = plan_shape(shape, true, nseq, &p);
  if (s != GDN_OK) return s;
  return run_fwd(p, cu_seqlens, q, k, v, g, beta, S0, o, S_final, nullptr, 0, workspace,
                 workspace_bytes, stream);
}

gdn_status gdn_varlen_bwd(const gdn_shape* shape, const int* cu_seqlens, int nseq,
                          const void* q, const void* k, const void* v, const void* g,
                          const void* beta, const float* S0, const void* dout,
                          const float* dS_final, void* dq, void* dk, void* dv, void* dg,
                          void* dbeta, float* dS0, void* workspace, size_t workspace_bytes,
                          void* stream) {
  Plan p;
  gdn_status s = plan_shape(shape, true, nseq, &p);
  if (s != GDN_OK) return s;
  return run_bwd(p, cu_seqlens, q, k, v, g, beta, S0, dout, dS_final, dq, dk, dv, dg, dbeta,
                 dS0, nullptr, 0, workspace, workspace_bytes, stream);
}

const char* gdn_status_str(gdn_status status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
  }
  return "GDN_ERR_UNKNOWN";
}

gdn_status gdn_workspace_status(void* workspace, void* stream) {
  if (!workspace || !al(workspace, kAlign)) return GDN_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GDN_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(workspace, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return GDN_ERR_CUDA;
  switch (word) {
    case DEV_OK: return GDN_OK;
    case DEV_BAD_CU_SEQLENS: return GDN_ERR_INVALID_ARG;
    case DEV_TIMEOUT: return GDN_ERR_TIMEOUT;
  }
  return GDN_ERR_CUDA;
}

int gdn_path(const gdn_shape* shape) {
  Plan p;
  if (plan_shape(shape, false, 0, &p) != GDN_OK) return 0;
  return path_of(p);
}

int gdn_version(void) { return 100; }

void gdn_profile_arm(void** events, int capacity) {
  gdn::g_prof_ev = (events && capacity > 0) ? (cudaEvent_t*)events : nullptr;
  gdn::g_prof_cap = capacity < 4096 ? capacity : 4096;
  gdn::g_prof_n = 0;
}

int gdn_profile_count(void) { return gdn::g_prof_n; }

int gdn_diag_wait_timeout(void* workspace, int limit_log2, void* stream) {
  if (!workspace || !al(workspace, kAlign)) return GDN_ERR_WORKSPACE;
  const int lg = limit_log2 < 10 ? 10 : (limit_log2 > 32 ? 32 : limit_log2);
  gdn::k_diag_wait<<<1, 32, 0, (cudaStream_t)stream>>>((int*)workspace, 1ll << lg);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

const char* gdn_profile_name(int i) {
  return (i >= 0 && i < gdn::g_prof_n) ? gdn::g_prof_names[i] : nullptr;
}

}  // extern "C"
