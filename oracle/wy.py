"""Chunkwise (WY) form of the gated delta rule in numpy fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

This is the second, independent CPU formulation. It follows the chunkwise
decomposition of a recurrent layer into Pre / ST / Out with the auxiliary
V^new (StateFlow review: referee report major comment 1, Eq. 2, and
"Assumptions & free parameters", Pre/ST/Out decomposition; kernel-level
chunking into blocks b_{i,j}), derived from the token recurrence of Gated Delta
Networks. Blocks are 64 tokens, anchored at the start of each sequence; a
shorter tail block is allowed. Per block, with local positions r = 1..C,
gamma_r = sum_{j<=r} g_j and Gamma_r = exp(gamma_r):

  Mask_{rj} = exp(gamma_r - gamma_j) for j <= r, else 0
  A  = strictly-lower( diag(beta) K K^T * Mask )          (Pre)
  T  = (I + A)^{-1}
  W  = T diag(beta * Gamma) K,   U = T diag(beta) V
  Vn = U - W H                                             (ST; V^new)
  H' = Gamma_C H + Kt^T Vn,      Kt_r = exp(gamma_C - gamma_r) k_r
  O  = diag(Gamma) Q H + (Q K^T * Mask) Vn                 (Out)

H is the state S^T (dk x dv). The backward pass is the reverse-mode derivative
of exactly these steps, block by block, with the states H_b re-created from
the chunk's input state (Eq. 6 of the review: Bwd rebuilds the trajectory Fwd
consumed, including V^new). Library primitives used: matmul and
``numpy.linalg.inv``.
"""
import numpy as np

BLOCK = 64


def _blocks(T, block=BLOCK):
    return [(s, min(T, s + block)) for s in range(0, T, block)]


def _block_terms(Kb, Vb, gb, bb):
    C = Kb.shape[0]
    gam = np.cumsum(gb)
    Gam = np.exp(gam)
    diff = gam[:, None] - gam[None, :]
    lower = np.tril(np.ones((C, C), dtype=bool))
    Mask = np.where(lower, np.exp(np.where(lower, diff, 0.0)), 0.0)
    A = np.tril(bb[:, None] * (Kb @ Kb.T) * Mask, -1)
    T = np.linalg.inv(np.eye(C) + A)
    W = T @ ((bb * Gam)[:, None] * Kb)
    U = T @ (bb[:, None] * Vb)
    decay_to_end = np.exp(gam[-1] - gam)
    return gam, Gam, Mask, A, T, W, U, decay_to_end


def _seq_fwd(Q, K, V, g, beta, H0):
    """One (sequence, head): Q [L, dk] ... Returns (O [L, dv], H_final, H_starts)."""
    L = Q.shape[0]
    H = H0.copy()
    O = np.zeros((L, V.shape[1]))
    starts = []
    for s, e in _blocks(L):
        starts.append(H.copy())
        gam, Gam, Mask, A, T, W, U, dte = _block_terms(K[s:e], V[s:e], g[s:e], beta[s:e])
        Vn = U - W @ H
        O[s:e] = Gam[:, None] * (Q[s:e] @ H) + ((Q[s:e] @ K[s:e].T) * Mask) @ Vn
        Kt = dte[:, None] * K[s:e]
        H = np.exp(gam[-1]) * H + Kt.T @ Vn
    return O, H, starts


def _seq_bwd(Q, K, V, g, beta, H0, dO, dH_end):
    L, dk = Q.shape
    dv = V.shape[1]
    _, _, starts = _seq_fwd(Q, K, V, g, beta, H0)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    dg = np.zeros_like(g)
    dbeta = np.zeros_like(beta)
    dH = dH_end.copy()
    for bi, (s, e) in reversed(list(enumerate(_blocks(L)))):
        Hb = starts[bi]
        Qb, Kb, Vb, gb, bb, dOb = Q[s:e], K[s:e], V[s:e], g[s:e], beta[s:e], dO[s:e]
        gam, Gam, Mask, A, T, W, U, dte = _block_terms(Kb, Vb, gb, bb)
        GamC = np.exp(gam[-1])
        Vn = U - W @ Hb
        Kt = dte[:, None] * Kb
        QK = Qb @ Kb.T
        QKM = QK * Mask
        # ST chain, reversed
        dVn = QKM.T @ dOb + Kt @ dH
        dHb = GamC * dH + (Gam[:, None] * Qb).T @ dOb - W.T @ dVn
        dgam = np.zeros(e - s)
        # Out: O = diag(Gamma) Q Hb + QKM Vn
        dOH = dOb @ Hb.T
        dQb = Gam[:, None] * dOH
        dgam += Gam * np.sum(Qb * dOH, axis=1)
        P = (dOb @ Vn.T) * Mask
        dQb += P @ Kb
        dKb = P.T @ Qb
        R = P * QK
        dgam += R.sum(axis=1) - R.sum(axis=0)
        # state update: H' = GamC Hb + Kt^T Vn
        dKt = Vn @ dH.T
        dKb += dte[:, None] * dKt
        rho = dte * np.sum(Kb * dKt, axis=1)
        dgam -= rho
        dgam[-1] += rho.sum() + GamC * np.sum(dH * Hb)
        # V^new = U - W Hb
        dU = dVn
        dW = -dVn @ Hb.T
        # W = T diag(beta Gamma) K, U = T diag(beta) V
        bG = bb * Gam
        dT = dW @ (bG[:, None] * Kb).T + dU @ (bb[:, None] * Vb).T
        X = T.T @ dW
        Y = T.T @ dU
        dKb += bG[:, None] * X
        xk = np.sum(X * Kb, axis=1)
        dbb = Gam * xk
        dgam += bG * xk
        dVb = bb[:, None] * Y
        dbb += np.sum(Y * Vb, axis=1)
        # T = (I + A)^{-1}
        dA = np.tril(-T.T @ dT @ T.T, -1)
        E = dA * Mask
        KK = Kb @ Kb.T
        dbb += np.sum(E * KK, axis=1)
        BE = bb[:, None] * E
        dKb += BE @ Kb + BE.T @ Kb
        G = dA * A
        dgam += G.sum(axis=1) - G.sum(axis=0)
        # gamma = cumsum(g) within the block
        dgb = np.cumsum(dgam[::-1])[::-1]
        dQ[s:e], dK[s:e], dV[s:e], dg[s:e], dbeta[s:e] = dQb, dKb, dVb, dgb, dbb
        dH = dHb
    return dQ, dK, dV, dg, dbeta, dH


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def fwd(q, k, v, g, beta, S_in=None):
    """Chunkwise forward, same contract as ``oracle.fwd``."""
    q, k, v, g, beta, S_in = map(_f64, (q, k, v, g, beta, S_in))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    S_out = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            H0 = S_in[b, h] if S_in is not None else np.zeros((dk, dv))
            o[b, :, h], S_out[b, h], _ = _seq_fwd(q[b, :, h], k[b, :, h], v[b, :, h],
                                                  g[b, :, h], beta[b, :, h], H0)
    return o, S_out


def bwd(q, k, v, g, beta, S_in, dout, dS_out=None):
    """Chunkwise backward, same contract as ``oracle.bwd``."""
    q, k, v, g, beta, S_in, dout, dS_out = map(_f64, (q, k, v, g, beta, S_in, dout, dS_out))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    outs = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(g),
            np.zeros_like(beta), np.zeros((B, H, dk, dv))]
    for b in range(B):
        for h in range(H):
            H0 = S_in[b, h] if S_in is not None else np.zeros((dk, dv))
            dHe = dS_out[b, h] if dS_out is not None else np.zeros((dk, dv))
            r = _seq_bwd(q[b, :, h], k[b, :, h], v[b, :, h], g[b, :, h], beta[b, :, h], H0,
                         dout[b, :, h], dHe)
            outs[0][b, :, h], outs[1][b, :, h], outs[2][b, :, h] = r[0], r[1], r[2]
            outs[3][b, :, h], outs[4][b, :, h], outs[5][b, h] = r[3], r[4], r[5]
    return tuple(outs)
