"""Parity where the arithmetic is most exposed, checked per head.

* The 256K-token, 16-head workload (8 chained chunks of 32768, the benchmark's
  launch configuration) with weak decay (alpha ~ 0.9995) and nonzero S_in /
  dS_out, so the fp32 state (and its bf16 copy used as an MMA operand) carries
  weight across all 4096 chained 64-token blocks.
* Ill-conditioned blocks: beta = 1 and near-collinear keys (with random
  signs) inside each 64-token block, the inputs that stress T = (I + A)^-1,
  whose off-diagonal blocks are formed with TF32 tensor-core MMAs.
* The packed variable-length workload at full size (dk 128, dv 256) with
  nonzero per-sequence initial states and final-state gradients, checking
  dS0 as well.

Every output is compared with the fp64 oracle per head (max-norm relative
error of each head against that head's own largest entry), which is stricter
than the whole-tensor figure for heads of small magnitude.
"""
import numpy as np
import pytest
import torch

import oracle
from chunked_linear_recurrence_gated_gb300 import gdn
from chunked_linear_recurrence_gated_gb300.inputs import cu_seqlens, make_inputs, workload
from helpers import BWD_TOL, FWD_TOL, GRAD_NAMES, np64, run_chunks_bwd, run_chunks_fwd

pytestmark = pytest.mark.gpu

BF = torch.bfloat16


def rel_err_per_head(got, ref, head_axis):
    """Max-norm relative error of every head: max|got - ref| / max|ref| over
    that head's entries."""
    got, ref = np64(got), np64(ref)
    got = np.moveaxis(got, head_axis, 0).reshape(got.shape[head_axis], -1)
    ref = np.moveaxis(ref, head_axis, 0).reshape(ref.shape[head_axis], -1)
    den = np.abs(ref).max(axis=1)
    num = np.abs(got - ref).max(axis=1)
    return [float(n / d) if d > 0 else float(n) for n, d in zip(num, den)]


def check_per_head(outs, refs, names, tols, head_axes):
    worst, bad = {}, []
    for name, got, ref, tol, ax in zip(names, outs, refs, tols, head_axes):
        errs = rel_err_per_head(got, ref, ax)
        worst[name] = max(errs)
        if worst[name] > tol:
            bad.append((name, errs, tol))
    print({k: f"{v:.2e}" for k, v in worst.items()})
    assert not bad, bad
    return worst


def test_long_weak_decay_chunked_parity_per_head():
    """256K tokens, H 16, d 128, bf16, 8 x 32768 chained chunks, weak decay,
    nonzero S_in and dS_out; heads 0 and 9 against the oracle."""
    d = make_inputs(1, 262144, 16, 128, 128, dtype=BF, seed=77, device="cuda", decay="weak",
                    do_scale=0.02, with_state=True)
    chunks = [32768] * 8
    o, S_out, S_ins = run_chunks_fwd(d, chunks, S_in=d["S_in"])
    grads = run_chunks_bwd(d, chunks, S_ins, dS_out=d["dS_out"])
    torch.cuda.synchronize()
    heads = [0, 9]
    x = {key: d[key][:, :, heads].float().cpu() for key in ("q", "k", "v", "g", "beta", "do")}
    S_in = d["S_in"][:, heads].cpu()
    dS_out = d["dS_out"][:, heads].cpu()
    o_ref, S_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S_in)
    g_ref = oracle.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S_in, x["do"], dS_out)
    outs = [o[:, :, heads], S_out[:, heads]] + [t[:, :, heads] for t in grads[:5]] + [grads[5][:, heads]]
    refs = [o_ref, S_ref] + list(g_ref)
    names = ["o", "S_out"] + GRAD_NAMES
    tols = [FWD_TOL[BF]] * 2 + [BWD_TOL[BF]] * 6
    axes = [2, 1, 2, 2, 2, 2, 2, 1]
    check_per_head(outs, refs, names, tols, axes)


def ill_conditioned_inputs(T, H, dtype, eps, seed):
    """beta = 1; in every 64-token block the keys are one unit direction with
    random signs plus eps-sized noise (renormalised); weak decay."""
    x = make_inputs(1, T, H, 128, 128, dtype=torch.float32, seed=seed, decay="weak",
                    with_state=True)
    gen = torch.Generator().manual_seed(seed + 1)
    k = torch.empty(1, T, H, 128)
    for b0 in range(0, T, 64):
        n = min(64, T - b0)
        base = torch.randn(1, 1, H, 128, generator=gen)
        base = base / base.norm(dim=-1, keepdim=True)
        sign = torch.where(torch.rand(1, n, H, 1, generator=gen) < 0.5, -1.0, 1.0)
        kk = sign * base + eps * torch.randn(1, n, H, 128, generator=gen)
        k[:, b0:b0 + n] = kk / kk.norm(dim=-1, keepdim=True)
    x["k"] = k
    x["beta"] = torch.ones(1, T, H)
    return {key: (t.to(dtype) if key not in ("S_in", "dS_out") else t) for key, t in x.items()}


# bf16 with keys collinear to within 1 % (cond(I + A) ~ 80): every bf16
# intermediate (T diag(beta Gamma), T diag(beta), W, U, V^new, the state
# operand) adds a 2^-9 relative rounding that the conditioning amplifies. A
# CPU emulation of those roundings reproduces the kernel's forward error on
# this input (2.5e-2) and shows that no single one dominates (dropping any one
# leaves 1.7e-2 to 2.2e-2), so the bound is scaled by 1.5 for this case only.
ADVERSARIAL_SCALE = {(BF, 1e-2): 1.5}


@pytest.mark.parametrize("dtype", [BF, torch.float32])
@pytest.mark.parametrize("eps", [1e-1, 1e-2])
def test_ill_conditioned_blocks(dtype, eps):
    x = ill_conditioned_inputs(320, 2, dtype, eps, seed=5)
    d = {key: t.cuda() for key, t in x.items()}
    o, S_out = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"])
    grads = gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"], d["do"],
                              d["dS_out"])
    torch.cuda.synchronize()
    c = {key: t.float() for key, t in x.items()}
    o_ref, S_ref = oracle.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["S_in"])
    g_ref = oracle.bwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["S_in"], c["do"], c["dS_out"])
    sc = ADVERSARIAL_SCALE.get((dtype, eps), 1.0)
    check_per_head([o, S_out] + list(grads), [o_ref, S_ref] + list(g_ref),
                   ["o", "S_out"] + GRAD_NAMES,
                   [sc * FWD_TOL[dtype]] * 2 + [sc * BWD_TOL[dtype]] * 6, [2, 1, 2, 2, 2, 2, 2, 1])


def test_varlen_full_size_with_state_gradients():
    """The packed workload (131072 tokens, H 16, dk 128, dv 256, 24 lognormal
    sequences) with per-sequence S0 and dS_final; heads 0 and 15, every
    output including dS0."""
    w = workload(4)
    nseq = len(w.seqlens)
    d = make_inputs(1, w.T, w.H, w.dk, w.dv, dtype=BF, seed=w.seed, device="cuda",
                    with_state=True, state_batch=nseq)
    cu = cu_seqlens(w.seqlens)
    o, Sf = gdn.gdn_varlen_fwd(cu.cuda(), d["q"], d["k"], d["v"], d["g"], d["beta"], S0=d["S_in"])
    grads = gdn.gdn_varlen_bwd(cu.cuda(), d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"],
                               d["do"], dS_final=d["dS_out"])
    torch.cuda.synchronize()
    heads = [0, 15]
    x = {key: d[key][:, :, heads].float().cpu() for key in ("q", "k", "v", "g", "beta", "do")}
    S0 = d["S_in"][:, heads].cpu()
    dSf = d["dS_out"][:, heads].cpu()
    o_ref, S_ref = oracle.varlen_fwd(cu, x["q"], x["k"], x["v"], x["g"], x["beta"], S0)
    g_ref = oracle.varlen_bwd(cu, x["q"], x["k"], x["v"], x["g"], x["beta"], S0, x["do"], dSf)
    outs = [o[:, :, heads], Sf[:, heads]] + [t[:, :, heads] for t in grads[:5]] + [grads[5][:, heads]]
    check_per_head(outs, [o_ref, S_ref] + list(g_ref), ["o", "S_final"] + GRAD_NAMES,
                   [FWD_TOL[BF]] * 2 + [BWD_TOL[BF]] * 6, [2, 1, 2, 2, 2, 2, 2, 1])
