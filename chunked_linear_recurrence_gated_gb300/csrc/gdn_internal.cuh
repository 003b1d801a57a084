// Internal launch interface between the C-ABI host code and the kernel files.
#pragma once

#include <cuda.h>

#include "gdn_common.cuh"

namespace gdn {

// fp32-arithmetic SIMT kernels (gdn_simt.cu).
size_t simt_max_smem();
cudaError_t simt_fwd(const SeqMap& m, int dk, int dv, int dtype, const void* q, const void* k,
                     const void* v, const void* g, const void* beta, const float* S_in,
                     void* o, float* S_out, const SimtWs& ws, cudaStream_t st);
cudaError_t simt_bwd(const SeqMap& m, int dk, int dv, int dtype, const void* q, const void* k,
                     const void* v, const void* g, const void* beta, const float* S_in,
                     const void* dout, const float* dS_out, void* dq, void* dk_out, void* dv_out,
                     void* dg, void* dbeta, float* dS_in, const SimtWs& ws, cudaStream_t st);

// bf16 tensor-core kernels; dk = 128, dv in {128, 256}.
// Pre (gdn_tc_pre.cu): W, U, QKM, padded K / Q, decay factors, T.
// nb > 0: only blocks [b0, b0 + nb) of each sequence (fixed-length calls).
// mark: record the kernel with the timing hook.
cudaError_t tc_pre(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const TcWs& ws, int b0, int nb,
                   cudaStream_t st, bool mark);
// Per-block gradients (gdn_tc_grad.cu).
cudaError_t tc_grad(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                    const void* beta, const void* dout, void* dq, void* dk_out, void* dv_out,
                    void* dg, void* dbeta, const TcWs& ws, cudaStream_t st);
// Whole forward / backward calls (gdn_tc_chain.cu). The backward skips the Pre
// kernel when run_pre is false: ws then points at Pre products (with T and
// K K^T) that a forward call wrote for the same inputs.
cudaError_t tc_fwd(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const float* S_in, void* o, float* S_out,
                   const TcWs& ws, const FwdSplit& sp, cudaStream_t st);
cudaError_t tc_bwd(const SeqMap& m, int dv, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const float* S_in, const void* dout,
                   const float* dS_out, void* dq, void* dk_out, void* dv_out, void* dg,
                   void* dbeta, float* dS_in, const TcWs& ws, bool run_pre, cudaStream_t st);

// Tensor maps for TMA copies (gdn_tc_pre.cu), 128-byte swizzle. make_tok_map
// views a [B][T][H][d] bf16 tensor (varlen: [1][total][H][d]) with
// 64-element x 1 head x 64-token boxes; make_ws_map a per-block-head
// workspace array [nbh][rows][row_stride] with 64-element x box_rows boxes.
cudaError_t make_tok_map(CUtensorMap* map, const void* base, int d, const SeqMap& m);
cudaError_t make_ws_map(CUtensorMap* map, const void* base, int inner, int rows, int row_stride,
                        long long nbh, int box_rows);

// Diagnostic timing hook (include/gdn_profile.h): records an event before the
// kernel named `next` (nullptr after the last kernel of a call) when armed.
void prof_mark(cudaStream_t st, const char* next);

// Builds the varlen block tables from device cu_seqlens (gdn_api.cu).
cudaError_t varlen_prep(const int* cu, int nseq, int T, int nblk_cap, int* blk0, int* blk_seq,
                        int* status, cudaStream_t st);

}  // namespace gdn
