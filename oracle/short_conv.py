"""fp64 oracle of the causal short convolution with carried boundary state.

TEST INFRASTRUCTURE ONLY (see the package docstring): tests, the smoke check
and the benchmark's CPU legs call it; the product never does.

The StateFlow review ("What carries the argument", and the footnote to its
Section 3.1 quoted in the referee report, major comment 1) says each chunk
carries, besides S_in / S_out, auxiliary local-convolution boundary states,
but prints no formula. Reading taken here (the causal depthwise short
convolution a Gated DeltaNet layer applies to its q / k / v projections):
for channel c, width W, weights w[c, 0..W-1], bias b[c] and the extended input
x_ext = [state_in ; x] (state_in holds the W - 1 inputs that precede the
chunk, zeros at a sequence start),

    z[t, c]   = b[c] + sum_j w[c, j] * x_ext[t + j, c]      (t = 0 .. T-1)
    y[t, c]   = act(z[t, c]),   act = identity or SiLU (z * sigmoid(z))
    state_out = x_ext[T .. T + W - 2]   (the last W - 1 inputs, raw)

so a sequence split into chunks with state_out -> next state_in reproduces
the unsplit convolution. The backward takes dy and d(state_out) and returns
dx, dw, db and d(state_in) (reverse-mode of the same definition).

Layouts: x, y [B, T, C]; states [B, W - 1, C] (token-major, like x);
w [C, W]; b [C].
"""
import numpy as np


def _ext(x, state_in, W):
    B, T, C = x.shape
    s = np.zeros((B, W - 1, C)) if state_in is None else np.asarray(state_in, np.float64)
    return np.concatenate([s, np.asarray(x, np.float64)], axis=1)


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def conv_fwd(x, w, b=None, state_in=None, act="silu"):
    """Returns (y, state_out) in fp64."""
    w = np.asarray(w, np.float64)
    C, W = w.shape
    xe = _ext(x, state_in, W)
    B, T = xe.shape[0], xe.shape[1] - (W - 1)
    z = np.zeros((B, T, C)) if b is None else np.broadcast_to(np.asarray(b, np.float64), (B, T, C)).copy()
    for j in range(W):
        z += w[:, j] * xe[:, j:j + T, :]
    y = z * _sigmoid(z) if act == "silu" else z
    return y, xe[:, T:T + W - 1, :].copy()


def conv_bwd(x, w, b, state_in, dy, dstate_out=None, act="silu"):
    """Returns (dx, dw, db, dstate_in) in fp64 for loss <dy, y> + <dstate_out, state_out>."""
    w = np.asarray(w, np.float64)
    C, W = w.shape
    xe = _ext(x, state_in, W)
    B, T = xe.shape[0], xe.shape[1] - (W - 1)
    z = np.zeros((B, T, C)) if b is None else np.broadcast_to(np.asarray(b, np.float64), (B, T, C)).copy()
    for j in range(W):
        z += w[:, j] * xe[:, j:j + T, :]
    dy = np.asarray(dy, np.float64)
    if act == "silu":
        s = _sigmoid(z)
        g = dy * s * (1.0 + z * (1.0 - s))
    else:
        g = dy
    dxe = np.zeros_like(xe)
    dw = np.zeros((C, W))
    for j in range(W):
        dxe[:, j:j + T, :] += w[:, j] * g
        dw[:, j] = (g * xe[:, j:j + T, :]).sum(axis=(0, 1))
    if dstate_out is not None:
        dxe[:, T:T + W - 1, :] += np.asarray(dstate_out, np.float64)
    db = g.sum(axis=(0, 1))
    return dxe[:, W - 1:, :], dw, db, dxe[:, :W - 1, :]
