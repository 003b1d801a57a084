"""Shared helpers for the GPU parity tests (comparison metrics, chunk loops)."""
import numpy as np
import torch

from chunked_linear_recurrence_gated_gb300 import gdn

FWD_TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
BWD_TOL = {torch.float32: 1e-3, torch.bfloat16: 3e-2}
GRAD_NAMES = ["dq", "dk", "dv", "dg", "dbeta", "dS_in"]


def np64(t):
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().float().cpu().double().numpy()


def rel_err(got, ref):
    """Max-norm relative error: max|got - ref| / max|ref| over the whole tensor."""
    got, ref = np64(got), np64(ref)
    den = np.abs(ref).max()
    if den == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / den)


def to_dev(x, dev="cuda"):
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}


def run_chunks_fwd(d, chunks, S_in=None):
    """Chained forward over chunk lengths (Eq. 5 chain). Returns (o, S_out, S_ins)."""
    outs, S_ins = [], []
    S = S_in
    t0 = 0
    for L in chunks:
        sl = slice(t0, t0 + L)
        S_ins.append(S)
        o, S = gdn.gdn_chunk_fwd(d["q"][:, sl].contiguous(), d["k"][:, sl].contiguous(),
                                 d["v"][:, sl].contiguous(), d["g"][:, sl].contiguous(),
                                 d["beta"][:, sl].contiguous(), S)
        outs.append(o)
        t0 += L
    return torch.cat(outs, dim=1), S, S_ins


def run_chunks_bwd(d, chunks, S_ins, dS_out=None):
    """Chained backward in reverse chunk order (Eq. 7 chain)."""
    parts = [None] * len(chunks)
    dS = dS_out
    starts = np.concatenate([[0], np.cumsum(chunks)[:-1]])
    for i in reversed(range(len(chunks))):
        sl = slice(int(starts[i]), int(starts[i]) + chunks[i])
        r = gdn.gdn_chunk_bwd(d["q"][:, sl].contiguous(), d["k"][:, sl].contiguous(),
                              d["v"][:, sl].contiguous(), d["g"][:, sl].contiguous(),
                              d["beta"][:, sl].contiguous(), S_ins[i], d["do"][:, sl].contiguous(),
                              dS)
        parts[i] = r[:5]
        dS = r[5]
    grads = [torch.cat([p[j] for p in parts], dim=1) for j in range(5)]
    return (*grads, dS)
