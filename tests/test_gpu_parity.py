"""GPU parity against the fp64 oracle through the C ABI: small shapes that span
several 64-token blocks and a ragged tail, edge cases, chunk-split bit-identity,
determinism, varlen, and the device-side status word."""
import numpy as np
import pytest
import torch

import oracle
from chunked_linear_recurrence_gated_gb300 import gdn
from chunked_linear_recurrence_gated_gb300.inputs import cu_seqlens, make_inputs, workload
from helpers import (BWD_TOL, FWD_TOL, GRAD_NAMES, rel_err, run_chunks_bwd, run_chunks_fwd,
                     to_dev)

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def check_against_oracle(x, dtype, chunks=None, tag=""):
    d = to_dev(x)
    T = x["q"].shape[1]
    chunks = chunks or [T]
    o, S_out, S_ins = run_chunks_fwd(d, chunks, d.get("S_in"))
    grads = run_chunks_bwd(d, chunks, S_ins, d.get("dS_out"))
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x.get("S_in"))
    g_ref = oracle.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x.get("S_in"), x["do"],
                       x.get("dS_out"))
    errs = {"o": rel_err(o, o_ref), "S_out": rel_err(S_out, S_ref)}
    for name, got, ref in zip(GRAD_NAMES, grads, g_ref):
        errs[name] = rel_err(got, ref)
    for name in ("o", "S_out"):
        assert errs[name] <= FWD_TOL[dtype], (tag, name, errs)
    for name in GRAD_NAMES:
        assert errs[name] <= BWD_TOL[dtype], (tag, name, errs)
    return errs


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (128, 256), (64, 128)])
@pytest.mark.parametrize("decay", ["default", "weak"])
def test_parity_small(dtype, dims, decay):
    dk, dv = dims
    x = make_inputs(2, 200, 3, dk, dv, dtype=DT[dtype], seed=dk + dv, decay=decay,
                    with_state=True)
    check_against_oracle(x, DT[dtype], tag=f"{dtype}-{dims}-{decay}")


@pytest.mark.parametrize("T", [1, 63, 64, 65, 129])
def test_parity_edge_lengths(T):
    for dtype in (torch.float32, torch.bfloat16):
        x = make_inputs(1, T, 2, 128, 128, dtype=dtype, seed=T, decay="weak", with_state=True)
        check_against_oracle(x, dtype, tag=f"T{T}")


def test_zero_state_arguments():
    """S_in = NULL and dS_out = NULL mean zero states."""
    x = make_inputs(1, 150, 2, 64, 64, dtype=torch.float32, seed=3)
    check_against_oracle(x, torch.float32)


def test_empty_chunk_passes_state_through():
    x = make_inputs(1, 1, 2, 128, 128, dtype=torch.bfloat16, seed=1, with_state=True)
    d = to_dev(x)
    e = {k: v[:, :0].contiguous() for k, v in d.items() if k not in ("S_in", "dS_out")}
    o, S_out = gdn.gdn_chunk_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], d["S_in"])
    r = gdn.gdn_chunk_bwd(e["q"], e["k"], e["v"], e["g"], e["beta"], d["S_in"], e["do"],
                          d["dS_out"])
    torch.cuda.synchronize()
    assert o.numel() == 0
    assert torch.equal(S_out, d["S_in"])
    assert torch.equal(r[5], d["dS_out"])


def test_tiny_fp32_exactness_workload():
    """Workload 0: B1 H2 T256 d64 fp32, two chained chunks of 128, S_in = 0."""
    w = workload(0)
    x = make_inputs(w.B, w.T, w.H, w.dk, w.dv, dtype=torch.float32, seed=w.seed)
    check_against_oracle(x, torch.float32, chunks=w.chunks, tag=w.name)


def run_full_and_split(x, chunks):
    d = to_dev(x)
    T = x["q"].shape[1]
    full_f = run_chunks_fwd(d, [T], d.get("S_in"))
    full_b = run_chunks_bwd(d, [T], full_f[2], d.get("dS_out"))
    split_f = run_chunks_fwd(d, chunks, d.get("S_in"))
    split_b = run_chunks_bwd(d, chunks, split_f[2], d.get("dS_out"))
    torch.cuda.synchronize()
    return full_f, full_b, split_f, split_b


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (128, 256)])
def test_split_bit_identical(dtype, dims):
    dk, dv = dims
    x = make_inputs(2, 448, 2, dk, dv, dtype=DT[dtype], seed=5, decay="weak", with_state=True)
    full_f, full_b, split_f, split_b = run_full_and_split(x, [64, 192, 128, 64])
    assert torch.equal(full_f[0], split_f[0])
    assert torch.equal(full_f[1], split_f[1])
    for a, b, name in zip(full_b, split_b, GRAD_NAMES):
        assert torch.equal(a, b), name


def test_split_with_ragged_tail_bit_identical():
    x = make_inputs(1, 300, 3, 128, 128, dtype=torch.bfloat16, seed=8, decay="weak",
                    with_state=True)
    full_f, full_b, split_f, split_b = run_full_and_split(x, [128, 172])
    assert torch.equal(full_f[0], split_f[0]) and torch.equal(full_f[1], split_f[1])
    for a, b in zip(full_b, split_b):
        assert torch.equal(a, b)


def test_deterministic():
    x = make_inputs(1, 640, 4, 128, 128, dtype=torch.bfloat16, seed=12, with_state=True)
    d = to_dev(x)
    a = run_chunks_fwd(d, [640], d["S_in"])
    ga = run_chunks_bwd(d, [640], a[2], d["dS_out"])
    b = run_chunks_fwd(d, [640], d["S_in"])
    gb = run_chunks_bwd(d, [640], b[2], d["dS_out"])
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for u, v in zip(ga, gb):
        assert torch.equal(u, v)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dims", [(128, 128), (128, 256), (64, 64)])
def test_varlen_parity(dtype, dims):
    dk, dv = dims
    lens = [64, 1, 130, 0, 200, 63]
    T = sum(lens)
    H = 2
    x = make_inputs(1, T, H, dk, dv, dtype=DT[dtype], seed=21, decay="weak", with_state=True,
                    state_batch=len(lens))
    cu = cu_seqlens(lens)
    d = to_dev(x)
    o, Sf = gdn.gdn_varlen_fwd(cu.cuda(), d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"])
    grads = gdn.gdn_varlen_bwd(cu.cuda(), d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"],
                               d["do"], d["dS_out"])
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.varlen_fwd(cu, x["q"], x["k"], x["v"], x["g"], x["beta"], x["S_in"])
    g_ref = oracle.varlen_bwd(cu, x["q"], x["k"], x["v"], x["g"], x["beta"], x["S_in"], x["do"],
                              x["dS_out"])
    tol_f, tol_b = FWD_TOL[DT[dtype]], BWD_TOL[DT[dtype]]
    assert rel_err(o, o_ref) <= tol_f
    assert rel_err(Sf, S_ref) <= tol_f
    for name, got, ref in zip(GRAD_NAMES, grads, g_ref):
        assert rel_err(got, ref) <= tol_b, name


def test_varlen_matches_fixed_length_bitwise():
    """A varlen call whose sequences all have length T equals the B = nseq fixed call."""
    B, T, H = 3, 200, 2
    x = make_inputs(B, T, H, 128, 128, dtype=torch.bfloat16, seed=4, decay="weak",
                    with_state=True)
    d = to_dev(x)
    o, S = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"])
    gr = gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"], d["do"],
                           d["dS_out"])
    flat = {k: (v.reshape(1, B * T, *v.shape[2:]) if k not in ("S_in", "dS_out") else v)
            for k, v in d.items()}
    cu = cu_seqlens([T] * B).cuda()
    o2, S2 = gdn.gdn_varlen_fwd(cu, flat["q"], flat["k"], flat["v"], flat["g"], flat["beta"],
                                d["S_in"])
    gr2 = gdn.gdn_varlen_bwd(cu, flat["q"], flat["k"], flat["v"], flat["g"], flat["beta"],
                             d["S_in"], flat["do"], d["dS_out"])
    torch.cuda.synchronize()
    assert torch.equal(o.reshape(o2.shape), o2) and torch.equal(S, S2)
    for a, b in zip(gr, gr2):
        assert torch.equal(a.reshape(b.shape), b)


def test_bad_cu_seqlens_reported_on_device():
    x = make_inputs(1, 256, 2, 128, 128, dtype=torch.bfloat16, seed=2)
    d = to_dev(x)
    bad = torch.tensor([0, 100, 50, 256], dtype=torch.int32, device="cuda")  # not monotone
    shape = gdn.shape_of(d["q"], d["v"])
    ws = gdn.alloc_workspace(gdn.varlen_workspace_bytes(shape, 3, False), "cuda")
    gdn.gdn_varlen_fwd(bad, d["q"], d["k"], d["v"], d["g"], d["beta"], workspace=ws)
    assert gdn.gdn_workspace_status(ws) == 1  # GDN_ERR_INVALID_ARG
    good = torch.tensor([0, 100, 150, 256], dtype=torch.int32, device="cuda")
    gdn.gdn_varlen_fwd(good, d["q"], d["k"], d["v"], d["g"], d["beta"], workspace=ws)
    assert gdn.gdn_workspace_status(ws) == 0
    short = torch.tensor([0, 100, 200], dtype=torch.int32, device="cuda")  # cu[nseq] != T
    gdn.gdn_varlen_fwd(short, d["q"], d["k"], d["v"], d["g"], d["beta"], workspace=ws)
    assert gdn.gdn_workspace_status(ws) == 1


def test_gpu_rejects_bad_calls_without_side_effects():
    x = make_inputs(1, 128, 2, 128, 128, dtype=torch.bfloat16, seed=2)
    d = to_dev(x)
    o = torch.full((1, 128, 2, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = gdn.alloc_workspace(256, "cuda")
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], o=o, workspace=ws)
    assert ei.value.status == 3
    torch.cuda.synchronize()
    assert (o.float() == 7.0).all()
