"""fp64 CPU oracle of the chunk-level gated delta rule.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers. The product path never imports this
package, and this package never imports the product (they share only the
seeded input generators, which hold none of the method's arithmetic).

Two independent formulations live here:

* ``fwd`` / ``bwd`` / ``varlen_fwd`` / ``varlen_bwd``: the token-by-token
  recurrence of the gated delta rule (Eq. 1 named in the StateFlow review,
  referee report major comment 1; written out as in Gated Delta Networks,
  reference [32] of that review) and its reverse-mode derivative, in C++ fp64
  (``gdn_oracle.cpp``). These are the parity oracle.
* ``wy``: the 64-token chunkwise form (Pre / ST / Out with the auxiliary
  V^new of Eq. 2, kernel-level blocks b_{i,j}) in numpy fp64, written from its
  derivation; the tests check it against the token loop, which pins the
  chunkwise algebra the GPU kernels implement.
* ``short_conv``: the causal short convolution with its carried boundary
  state (the auxiliary local-convolution states of the StateFlow review) and
  its reverse-mode derivative, numpy fp64.

Array layouts: q, k [B, T, H, dk]; v, o [B, T, H, dv]; g, beta [B, T, H];
states [B, H, dk, dv] holding S^T (o_t = state^T q_t). Varlen: B = 1 and
``cu_seqlens`` (int32, length nseq + 1) splits the T tokens into sequences;
states are [nseq, H, dk, dv].
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.gdn_oracle_fwd.argtypes = [I, I, I, I, I] + [P] * 8 + [I]
        lib.gdn_oracle_bwd.argtypes = [I, I, I, I, I] + [P] * 14 + [I]
        lib.gdn_oracle_varlen_fwd.argtypes = [I, I, I, P, I] + [P] * 8 + [I]
        lib.gdn_oracle_varlen_bwd.argtypes = [I, I, I, P, I] + [P] * 14 + [I]
        for f in (lib.gdn_oracle_fwd, lib.gdn_oracle_bwd,
                  lib.gdn_oracle_varlen_fwd, lib.gdn_oracle_varlen_bwd):
            f.restype = I
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def fwd(q, k, v, g, beta, S_in=None, nthreads=None):
    """Forward of one chunk per batch row. Returns (o, S_out), float64."""
    q, k, v, g, beta, S_in = map(_f64, (q, k, v, g, beta, S_in))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    S_out = np.zeros((B, H, dk, dv))
    rc = _load().gdn_oracle_fwd(B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                _ptr(beta), _ptr(S_in), _ptr(o), _ptr(S_out),
                                nthreads or default_threads())
    if rc:
        raise ValueError("gdn_oracle_fwd: invalid arguments")
    return o, S_out


def bwd(q, k, v, g, beta, S_in, dout, dS_out=None, nthreads=None):
    """Backward of one chunk for the loss <dout, o> + <dS_out, S_out>.

    Returns (dq, dk, dv, dg, dbeta, dS_in), float64.
    """
    q, k, v, g, beta, S_in, dout, dS_out = map(_f64, (q, k, v, g, beta, S_in, dout, dS_out))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dq = np.zeros_like(q)
    dk_ = np.zeros_like(k)
    dv_ = np.zeros_like(v)
    dg = np.zeros_like(g)
    dbeta = np.zeros_like(beta)
    dS_in = np.zeros((B, H, dk, dv))
    rc = _load().gdn_oracle_bwd(B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                _ptr(beta), _ptr(S_in), _ptr(dout), _ptr(dS_out),
                                _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg), _ptr(dbeta),
                                _ptr(dS_in), nthreads or default_threads())
    if rc:
        raise ValueError("gdn_oracle_bwd: invalid arguments")
    return dq, dk_, dv_, dg, dbeta, dS_in


def _cu(cu_seqlens):
    if hasattr(cu_seqlens, "detach"):
        cu_seqlens = cu_seqlens.detach().cpu().numpy()
    return np.ascontiguousarray(cu_seqlens, dtype=np.int32)


def varlen_fwd(cu_seqlens, q, k, v, g, beta, S0=None, nthreads=None):
    """Packed variable-length forward (B = 1). Returns (o, S_final [nseq,H,dk,dv])."""
    cu = _cu(cu_seqlens)
    q, k, v, g, beta, S0 = map(_f64, (q, k, v, g, beta, S0))
    _, T, H, dk = q.shape
    dv = v.shape[-1]
    nseq = len(cu) - 1
    o = np.zeros((1, T, H, dv))
    S_final = np.zeros((nseq, H, dk, dv))
    rc = _load().gdn_oracle_varlen_fwd(H, dk, dv, _ptr(cu), nseq, _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(g), _ptr(beta), _ptr(S0), _ptr(o), _ptr(S_final),
                                       nthreads or default_threads())
    if rc:
        raise ValueError("gdn_oracle_varlen_fwd: invalid arguments")
    return o, S_final


def varlen_bwd(cu_seqlens, q, k, v, g, beta, S0, dout, dS_final=None, nthreads=None):
    """Packed variable-length backward. Returns (dq, dk, dv, dg, dbeta, dS0)."""
    cu = _cu(cu_seqlens)
    q, k, v, g, beta, S0, dout, dS_final = map(_f64, (q, k, v, g, beta, S0, dout, dS_final))
    _, T, H, dk = q.shape
    dv = v.shape[-1]
    nseq = len(cu) - 1
    dq = np.zeros_like(q)
    dk_ = np.zeros_like(k)
    dv_ = np.zeros_like(v)
    dg = np.zeros_like(g)
    dbeta = np.zeros_like(beta)
    dS0 = np.zeros((nseq, H, dk, dv))
    rc = _load().gdn_oracle_varlen_bwd(H, dk, dv, _ptr(cu), nseq, _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(g), _ptr(beta), _ptr(S0), _ptr(dout),
                                       _ptr(dS_final), _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg),
                                       _ptr(dbeta), _ptr(dS0), nthreads or default_threads())
    if rc:
        raise ValueError("gdn_oracle_varlen_bwd: invalid arguments")
    return dq, dk_, dv_, dg, dbeta, dS0
