/*
 * gdn.h -- C ABI of the GB300 chunk-level Gated DeltaNet state transition.
 *
 * What the library computes
 * -------------------------
 * One call processes one sequence chunk C_i of a long sequence (StateFlow
 * review, "What carries the argument"): it takes the compact boundary state
 * S_i^in and the chunk's per-token q, k, v, log-decay g and write strength
 * beta, and returns the outputs o and S_i^out through the gated delta rule
 * (Eq. 1 named in the review's referee report, major comment 1; the form of
 * Gated Delta Networks, reference [32] of that review):
 *
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = S_t q_t,        alpha_t = exp(g_t).
 *
 * It is evaluated in 64-token blocks (the kernel-level blocks b_{i,j} of the
 * review's "Assumptions & free parameters") with the chunkwise Pre / ST / Out
 * decomposition and the auxiliary V^new (Eq. 2). The backward call takes
 * do and dS_out and returns dq, dk, dv, dg, dbeta and dS_in for the loss
 * <do, o> + <dS_out, S_out>, recomputing the chunk's trajectory from S_in
 * (Eq. 6). Chaining the calls gives the review's forward chain
 * S_{i+1}^in = S_i^out (Eq. 5) and backward chain dS_i^out = dS_{i+1}^in
 * (Eq. 7); with chunk boundaries at multiples of 64 tokens the chained
 * results are bit-identical to one call over the whole sequence.
 *
 * Conventions
 * -----------
 * - No q scaling and no normalisation inside: the caller normalises q, k and
 *   applies the sigmoid / log-decay maps. g is the log-decay (alpha = e^g),
 *   beta is already in (0, 1).
 * - Layouts (contiguous, row-major):
 *     q, k, dq, dk          [B, T, H, dk]
 *     v, o, do, dv          [B, T, H, dv]
 *     g, beta, dg, dbeta    [B, T, H]
 *     S_in, S_out, dS_*     [B, H, dk, dv] fp32; element [i][j] multiplies
 *                           q[i] into o[j], i.e. the state is stored as S^T.
 *   Varlen calls use B = 1, T = total tokens, and states [nseq, H, dk, dv].
 * - dtype: GDN_DTYPE_F32 or GDN_DTYPE_BF16 for q, k, v, g, beta, o and all
 *   input gradients; states and state gradients are always fp32.
 * - Supported sizes: dk in {64, 128}, dv in {64, 128, 256}, H >= 1, B >= 1,
 *   T >= 0. A tail block shorter than 64 tokens is handled by masking.
 * - Alignment: every tensor pointer must be 16-byte aligned; the workspace
 *   must be 256-byte aligned.
 *
 * Ownership and execution
 * -----------------------
 * The caller owns every buffer, including the workspace (size from the
 * *_workspace_bytes functions). The library allocates no device memory and
 * keeps no state between calls other than per-device kernel attributes (and
 * the fixed scratch array of gdn_chunk_fwd_noalloc, below).
 * All work is enqueued on `stream` (a cudaStream_t passed as void*, NULL =
 * the legacy default stream); calls return without synchronising. S_out may
 * alias S_in and dS_in may alias dS_out. Other outputs must not alias
 * inputs. Concurrent calls must use distinct workspaces.
 *
 * Errors
 * ------
 * Every argument is checked on the host before anything is launched; a bad
 * argument returns GDN_ERR_INVALID_ARG / GDN_ERR_UNSUPPORTED /
 * GDN_ERR_WORKSPACE and leaves every buffer untouched. A launch failure
 * returns GDN_ERR_CUDA. Kernels never trap. Conditions that only the device
 * can see (a malformed cu_seqlens array, a bounded wait that gave up) are
 * recorded in a status word in the workspace and the affected work is
 * skipped; gdn_workspace_status reads it (gdn_noalloc_status for
 * gdn_chunk_fwd_noalloc, whose status word sits in the library's scratch).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1, /* null pointer, negative size, misalignment, bad cu_seqlens */
  GDN_ERR_UNSUPPORTED = 2, /* dk / dv / dtype outside the supported set */
  GDN_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or too small */
  GDN_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  GDN_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up */
} gdn_status;

typedef enum { GDN_DTYPE_F32 = 0, GDN_DTYPE_BF16 = 1 } gdn_dtype;

typedef struct {
  int B;     /* batch (sequences); 1 for varlen calls */
  int T;     /* tokens per sequence in this chunk; total tokens for varlen calls */
  int H;     /* heads */
  int dk;    /* key / query head dimension */
  int dv;    /* value head dimension */
  int dtype; /* gdn_dtype */
} gdn_shape;

/* Workspace bytes needed by gdn_chunk_fwd (is_bwd = 0), gdn_chunk_bwd
 * (is_bwd = 1), or gdn_chunk_fwd_save / gdn_chunk_bwd_saved (is_bwd =
 * GDN_WS_SAVED) for `shape`; 0 if the shape is invalid or unsupported. */
#define GDN_WS_SAVED 2
size_t gdn_chunk_workspace_bytes(const gdn_shape* shape, int is_bwd);

/* Forward of one chunk (Eq. 5 chain: pass S_out as the next chunk's S_in).
 * S_in: NULL means a zero initial state. S_out: NULL skips writing it. */
gdn_status gdn_chunk_fwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, const float* S_in, void* o,
                         float* S_out, void* workspace, size_t workspace_bytes, void* stream);

/* Backward of one chunk (Eq. 6 recompute from S_in; Eq. 7 chain: pass dS_in
 * as the previous chunk's dS_out). S_in / dS_out: NULL means zero.
 * dS_in: NULL skips writing it. */
gdn_status gdn_chunk_bwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, const float* S_in, const void* dout,
                         const float* dS_out, void* dq, void* dk, void* dv, void* dg,
                         void* dbeta, float* dS_in, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Forward + backward that keep the forward's per-block products. The
 * backward rebuilds the trajectory from S_in (Eq. 6); its first step is the
 * same per-block Pre work (Eq. 2's decay cumsums, the masked K K^T / Q K^T,
 * T = (I + A)^-1, W and U) that the forward already did on the same inputs.
 * gdn_chunk_fwd_save computes exactly what gdn_chunk_fwd computes and also
 * leaves those products (plus T and the masked K K^T the gradient needs) and
 * the chain's per-block state H_b and V^new (bf16) in `saved`;
 * gdn_chunk_bwd_saved, given the same shape and inputs, reads them there
 * instead of recomputing them (only the reverse chain and the gradient kernel
 * run), and its results are bit-identical to gdn_chunk_bwd's. `saved` is a caller-owned device buffer of
 * gdn_chunk_saved_bytes(shape) bytes, 256-byte aligned, that must not change
 * between the two calls; `workspace` is gdn_chunk_workspace_bytes(shape,
 * GDN_WS_SAVED) bytes (the same buffer can serve both calls). A null,
 * misaligned or short `saved` returns GDN_ERR_WORKSPACE. Passing products of
 * other inputs is not detected and gives the gradient of neither. For shapes
 * on the fp32 kernels nothing is kept (gdn_chunk_saved_bytes returns 256)
 * and the backward recomputes as gdn_chunk_bwd does. */
size_t gdn_chunk_saved_bytes(const gdn_shape* shape);

gdn_status gdn_chunk_fwd_save(const gdn_shape* shape, const void* q, const void* k,
                              const void* v, const void* g, const void* beta, const float* S_in,
                              void* o, float* S_out, void* saved, size_t saved_bytes,
                              void* workspace, size_t workspace_bytes, void* stream);

gdn_status gdn_chunk_bwd_saved(const gdn_shape* shape, const void* q, const void* k,
                               const void* v, const void* g, const void* beta,
                               const float* S_in, const void* dout, const float* dS_out,
                               void* dq, void* dk, void* dv, void* dg, void* dbeta, float* dS_in,
                               const void* saved, size_t saved_bytes, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Varlen (packed) variants: B must be 1 and T is the total token count.
 * cu_seqlens is a DEVICE int32 array of nseq + 1 offsets with cu[0] = 0,
 * non-decreasing, cu[nseq] = T. The recurrence restarts at every sequence
 * start from S0[s] (NULL = zero) and the block grid is anchored there. */
size_t gdn_varlen_workspace_bytes(const gdn_shape* shape, int nseq, int is_bwd);

gdn_status gdn_varlen_fwd(const gdn_shape* shape, const int* cu_seqlens, int nseq,
                          const void* q, const void* k, const void* v, const void* g,
                          const void* beta, const float* S0, void* o, float* S_final,
                          void* workspace, size_t workspace_bytes, void* stream);

gdn_status gdn_varlen_bwd(const gdn_shape* shape, const int* cu_seqlens, int nseq,
                          const void* q, const void* k, const void* v, const void* g,
                          const void* beta, const float* S0, const void* dout,
                          const float* dS_final, void* dq, void* dk, void* dv, void* dg,
                          void* dbeta, float* dS0, void* workspace, size_t workspace_bytes,
                          void* stream);

/* gdn_chunk_fwd without a caller-provided workspace. (No counterpart on the
 * StateFlow pages: this serves callers that cannot allocate device memory,
 * e.g. code running under a host framework that owns all device memory and
 * offers no allocator, or code that must not trigger an allocation while it
 * runs.) Arguments and results are those of gdn_chunk_fwd. The scratch is a
 * library-owned device array of GDN_NOALLOC_SCRATCH_BYTES, held by every GPU
 * that loads the library until the process exits; a shape whose forward
 * workspace (gdn_chunk_workspace_bytes(shape, 0)) exceeds it is rejected with
 * GDN_ERR_WORKSPACE before anything is launched (for dk = dv = 128 bf16 the
 * forward workspace is 77 KiB per 64-token block and head plus 128 KiB per
 * sequence and head, so the limit is B * ceil(T / 64) * H <= 849 for B = H = 1
 * and <= 816 for B = 1, H = 16). The call
 * allocates nothing. Its first call on a device looks up the array's device
 * address on the current device; make that first call before any stream
 * capture. Every call on a device shares the one array and no part of it needs
 * to start at zero; calls whose GPU work overlaps (other streams, other host
 * threads) race on it and must be serialised by the caller. */
#define GDN_NOALLOC_SCRATCH_BYTES (64u << 20)
gdn_status gdn_chunk_fwd_noalloc(const gdn_shape* shape, const void* q, const void* k,
                                 const void* v, const void* g, const void* beta,
                                 const float* S_in, void* o, float* S_out, void* stream);

/* The device-side status of gdn_chunk_fwd_noalloc calls on the current device
 * (what gdn_workspace_status reports for a caller-provided workspace): a
 * bounded wait that gave up inside the last call leaves GDN_ERR_TIMEOUT, and
 * that call's outputs are then incomplete. Synchronises `stream`, returns the
 * recorded status (GDN_OK if none) and resets it. Allocates nothing. The
 * scratch array's device address is cached per device and context; it is
 * looked up again after a device reset. */
gdn_status gdn_noalloc_status(void* stream);

/* Human-readable name of a status code (static string). */
const char* gdn_status_str(gdn_status status);

/* Synchronises `stream`, then returns the device-side status recorded in
 * `workspace` by the last call that used it (GDN_OK if nothing was
 * recorded). Resets the word to GDN_OK. */
gdn_status gdn_workspace_status(void* workspace, void* stream);

/* Which kernel family serves `shape` (0 = none / unsupported,
 * 1 = fp32 SIMT kernels, 2 = bf16 tensor-core kernels). Depends only on
 * dtype, dk and dv, never on T. */
int gdn_path(const gdn_shape* shape);

/* ABI version (major * 100 + minor). */
int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
