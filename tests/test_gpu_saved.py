"""Forward-products reuse (gdn_chunk_fwd_save / gdn_chunk_bwd_saved) through the
C ABI: every output bit-identical to the recomputing calls, chained over
chunks, and within tolerance of the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from chunked_linear_recurrence_gated_gb300 import gdn
from chunked_linear_recurrence_gated_gb300.inputs import make_inputs
from helpers import BWD_TOL, FWD_TOL, GRAD_NAMES, rel_err, run_chunks_bwd, run_chunks_fwd, to_dev

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def run_saved(d, chunks):
    """Chained forward keeping products, then chained backward reading them."""
    starts = np.concatenate([[0], np.cumsum(chunks)[:-1]]).astype(int)
    cut = lambda name, i: d[name][:, starts[i]:starts[i] + chunks[i]].contiguous()
    outs, S_ins, saved = [], [], []
    S = d.get("S_in")
    for i in range(len(chunks)):
        S_ins.append(S)
        o, S, sv = gdn.gdn_chunk_fwd_save(cut("q", i), cut("k", i), cut("v", i), cut("g", i),
                                          cut("beta", i), S)
        outs.append(o)
        saved.append(sv)
    parts = [None] * len(chunks)
    dS = d.get("dS_out")
    for i in reversed(range(len(chunks))):
        r = gdn.gdn_chunk_bwd_saved(cut("q", i), cut("k", i), cut("v", i), cut("g", i),
                                    cut("beta", i), S_ins[i], cut("do", i), saved[i], dS)
        parts[i] = r[:5]
        dS = r[5]
    grads = [torch.cat([p[j] for p in parts], dim=1) for j in range(5)]
    return torch.cat(outs, dim=1), S, grads + [dS]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (128, 256)])
def test_saved_matches_recompute_bitwise(dtype, dims):
    dk, dv = dims
    x = make_inputs(2, 200, 3, dk, dv, dtype=DT[dtype], seed=31 + dk + dv, decay="weak",
                    with_state=True)
    d = to_dev(x)
    chunks = [136, 64]
    o_a, S_a, S_ins = run_chunks_fwd(d, chunks, d["S_in"])
    g_a = run_chunks_bwd(d, chunks, S_ins, d["dS_out"])
    o_b, S_b, g_b = run_saved(d, chunks)
    torch.cuda.synchronize()
    assert torch.equal(o_a, o_b) and torch.equal(S_a, S_b)
    for a, b, name in zip(g_a, g_b, GRAD_NAMES):
        assert torch.equal(a, b), name


def test_saved_against_oracle_ragged():
    x = make_inputs(1, 333, 2, 128, 128, dtype=torch.bfloat16, seed=77, with_state=True)
    d = to_dev(x)
    o, S, grads = run_saved(d, [192, 141])
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S_in"])
    g_ref = oracle.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S_in"], x["do"],
                       x["dS_out"])
    assert rel_err(o, o_ref) <= FWD_TOL[torch.bfloat16]
    assert rel_err(S, S_ref) <= FWD_TOL[torch.bfloat16]
    for name, got, ref in zip(GRAD_NAMES, grads, g_ref):
        assert rel_err(got, ref) <= BWD_TOL[torch.bfloat16], name


def test_saved_shared_workspace_and_empty_chunk():
    """One workspace serves both calls; an empty chunk passes the states through."""
    x = make_inputs(1, 130, 2, 128, 128, dtype=torch.bfloat16, seed=4, with_state=True)
    d = to_dev(x)
    s = gdn.shape_of(d["q"], d["v"])
    ws = gdn.alloc_workspace(gdn.chunk_workspace_bytes(s, gdn.GDN_WS_SAVED), "cuda")
    o, S, sv = gdn.gdn_chunk_fwd_save(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"],
                                      workspace=ws)
    r = gdn.gdn_chunk_bwd_saved(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"], d["do"],
                                sv, d["dS_out"], workspace=ws)
    o2, S2 = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"])
    r2 = gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"], d["do"],
                           d["dS_out"])
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(S, S2)
    for a, b in zip(r, r2):
        assert torch.equal(a, b)
    e = {k: v[:, :0].contiguous() for k, v in d.items() if k not in ("S_in", "dS_out")}
    oe, Se, sve = gdn.gdn_chunk_fwd_save(e["q"], e["k"], e["v"], e["g"], e["beta"], d["S_in"])
    re_ = gdn.gdn_chunk_bwd_saved(e["q"], e["k"], e["v"], e["g"], e["beta"], d["S_in"], e["do"],
                                  sve, d["dS_out"])
    torch.cuda.synchronize()
    assert oe.numel() == 0 and torch.equal(Se, d["S_in"]) and torch.equal(re_[5], d["dS_out"])
