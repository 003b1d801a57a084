/*
 * gdn_conv.h -- C ABI of the causal short convolution with carried boundary
 * state (part of libgdn.so; status codes and dtypes from gdn.h).
 *
 * What it computes
 * ----------------
 * Besides S_in / S_out, each chunk of a Gated DeltaNet layer carries
 * auxiliary local-convolution boundary states (StateFlow review, "What
 * carries the argument", and the footnote to its Section 3.1 quoted in the
 * referee report, major comment 1). The pages give no formula; the reading
 * implemented here is the causal depthwise short convolution such a layer
 * applies to its q / k / v projections before the recurrence. For channel c,
 * width W, weights w[c][0..W-1], bias b[c] and the extended input
 * x_ext = [state_in ; x] (state_in = the W - 1 inputs preceding the chunk):
 *
 *     z[t][c]   = b[c] + sum_{j<W} w[c][j] * x_ext[t + j][c],   t = 0 .. T-1
 *     y[t][c]   = act(z[t][c]),   act = identity or SiLU (z * sigmoid(z))
 *     state_out = x_ext[T .. T + W - 2]      (the last W - 1 raw inputs)
 *
 * so chaining state_out -> next chunk's state_in reproduces the unsplit
 * convolution bit for bit (y and states). The backward returns, for the loss
 * <dy, y> + <dstate_out, state_out>, dx, dw, db and dstate_in; dstate_in is
 * the previous chunk's dstate_out. dw and db are this chunk's sums over B and
 * T (the caller adds the chunks' contributions).
 *
 * Conventions
 * -----------
 * - Layouts (contiguous, row-major): x, y, dy, dx [B, T, C]; state_in,
 *   state_out, dstate_* [B, W - 1, C] (token-major like x, same dtype as x);
 *   w, dw [C, W] fp32; b, db [C] fp32.
 * - dtype: GDN_DTYPE_F32 or GDN_DTYPE_BF16 for x, y, states and their
 *   gradients; arithmetic is fp32.
 * - Sizes: B >= 1, T >= 0, 2 <= W <= 8, C >= 1 a multiple of 4.
 * - Alignment: x, y, dy, dx and the states 16-byte aligned; w, b, dw, db
 *   4-byte aligned; the workspace 256-byte aligned.
 * - Outputs must not alias inputs (state_out must not alias state_in).
 * - NULL state_in means zeros (a sequence start); NULL state_out /
 *   dstate_in skip writing them; NULL dstate_out means zero; NULL b means no
 *   bias (then db may be NULL too).
 *
 * Ownership, execution and errors as in gdn.h: caller-owned buffers, work
 * enqueued on `stream` without synchronising, every argument checked on the
 * host before any launch (GDN_ERR_INVALID_ARG / GDN_ERR_UNSUPPORTED /
 * GDN_ERR_WORKSPACE), GDN_ERR_CUDA if a launch fails. The forward needs no
 * workspace; the backward's holds per-tile partial sums of dw and db, reduced
 * in a fixed order (the results are deterministic).
 */
#ifndef GDN_CONV_H_
#define GDN_CONV_H_

#include <stddef.h>

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_CONV_ACT_NONE 0
#define GDN_CONV_ACT_SILU 1

typedef struct {
  int B;     /* sequences */
  int T;     /* tokens per sequence in this chunk */
  int C;     /* channels */
  int W;     /* kernel width (2..8) */
  int dtype; /* gdn_dtype of x, y, states */
  int act;   /* GDN_CONV_ACT_NONE or GDN_CONV_ACT_SILU */
} gdn_conv_shape;

/* Workspace bytes of gdn_conv_bwd for `shape`; 0 if the shape is invalid or
 * unsupported. */
size_t gdn_conv_workspace_bytes(const gdn_conv_shape* shape);

/* Forward of one chunk: y and state_out from x, w, b and state_in. */
gdn_status gdn_conv_fwd(const gdn_conv_shape* shape, const void* x, const float* w,
                        const float* b, const void* state_in, void* y, void* state_out,
                        void* stream);

/* Backward of one chunk: dx, dw, db and dstate_in from dy and dstate_out
 * (recomputes z from x, w, b and state_in). */
gdn_status gdn_conv_bwd(const gdn_conv_shape* shape, const void* x, const float* w,
                        const float* b, const void* state_in, const void* dy,
                        const void* dstate_out, void* dx, float* dw, float* db, void* dstate_in,
                        void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_CONV_H_ */
