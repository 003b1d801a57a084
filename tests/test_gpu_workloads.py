"""The four bf16 workloads at full size, in the launch configuration the
benchmark times (one gdn_chunk_* call per chunk, states chained), compared with
the fp64 oracle on sampled heads, plus chunk-split bit-identity against one
unsplit call.

Sampled heads keep the oracle to tens of seconds: the heads are independent
problems, so checking a head checks every output the oracle can produce for it.
"""
import numpy as np
import pytest
import torch

import oracle
from chunked_linear_recurrence_gated_gb300 import gdn
from chunked_linear_recurrence_gated_gb300.inputs import cu_seqlens, make_workload_inputs, workload
from helpers import BWD_TOL, FWD_TOL, GRAD_NAMES, rel_err, run_chunks_bwd, run_chunks_fwd

pytestmark = pytest.mark.gpu

BF = torch.bfloat16


def heads_of(x, heads):
    out = {}
    for key in ("q", "k", "v", "g", "beta", "do"):
        out[key] = x[key][:, :, heads].float().cpu()
    return out


def check_heads(w, d, o, S_out, grads, heads):
    x = heads_of(d, heads)
    o_ref, S_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], None)
    g_ref = oracle.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], None, x["do"], None)
    errs = {"o": rel_err(o[:, :, heads], o_ref), "S_out": rel_err(S_out[:, heads], S_ref)}
    for name, got, ref in zip(GRAD_NAMES[:5], grads[:5], g_ref[:5]):
        errs[name] = rel_err(got[:, :, heads], ref)
    errs["dS_in"] = rel_err(grads[5][:, heads], g_ref[5])
    print(w.name, {k: f"{v:.2e}" for k, v in errs.items()})
    for k_ in ("o", "S_out"):
        assert errs[k_] <= FWD_TOL[BF], (k_, errs)
    for k_ in GRAD_NAMES:
        assert errs[k_] <= BWD_TOL[BF], (k_, errs)


@pytest.mark.parametrize("index,heads", [(1, list(range(16))), (2, [0, 9]), (3, [0, 31])])
def test_chunked_workload_parity(index, heads):
    w = workload(index)
    d = make_workload_inputs(w, device="cuda")
    o, S_out, S_ins = run_chunks_fwd(d, w.chunks)
    grads = run_chunks_bwd(d, w.chunks, S_ins)
    torch.cuda.synchronize()
    check_heads(w, d, o, S_out, grads, heads)


@pytest.mark.parametrize("index", [1, 2, 3])
def test_chunked_workload_bit_identical_to_unsplit(index):
    w = workload(index)
    d = make_workload_inputs(w, device="cuda")
    o, S_out, S_ins = run_chunks_fwd(d, w.chunks)
    grads = run_chunks_bwd(d, w.chunks, S_ins)
    o1, S1, S_ins1 = run_chunks_fwd(d, [w.T])
    grads1 = run_chunks_bwd(d, [w.T], S_ins1)
    torch.cuda.synchronize()
    assert torch.equal(o, o1)
    assert torch.equal(S_out, S1)
    for a, b, name in zip(grads, grads1, GRAD_NAMES):
        assert torch.equal(a, b), name


def test_varlen_workload_parity():
    w = workload(4)
    d = make_workload_inputs(w, device="cuda")
    cu = cu_seqlens(w.seqlens)
    o, Sf = gdn.gdn_varlen_fwd(cu.cuda(), d["q"], d["k"], d["v"], d["g"], d["beta"])
    grads = gdn.gdn_varlen_bwd(cu.cuda(), d["q"], d["k"], d["v"], d["g"], d["beta"], None,
                               d["do"])
    torch.cuda.synchronize()
    heads = [0, 15]
    x = heads_of(d, heads)
    o_ref, S_ref = oracle.varlen_fwd(cu, x["q"], x["k"], x["v"], x["g"], x["beta"])
    g_ref = oracle.varlen_bwd(cu, x["q"], x["k"], x["v"], x["g"], x["beta"], None, x["do"])
    errs = {"o": rel_err(o[:, :, heads], o_ref), "S_final": rel_err(Sf[:, heads], S_ref)}
    for name, got, ref in zip(GRAD_NAMES[:5], grads[:5], g_ref[:5]):
        errs[name] = rel_err(got[:, :, heads], ref)
    print(w.name, {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["o"] <= FWD_TOL[BF] and errs["S_final"] <= FWD_TOL[BF], errs
    for name in GRAD_NAMES[:5]:
        assert errs[name] <= BWD_TOL[BF], (name, errs)
    # every sequence restarts from a zero state: splitting the packed batch at a
    # sequence boundary into two varlen calls gives bit-identical results
    cut = len(w.seqlens) // 2
    t_cut = int(cu[cut])
    parts = []
    for lo, hi, lens in ((0, t_cut, w.seqlens[:cut]), (t_cut, w.T, w.seqlens[cut:])):
        sub = {k_: d[k_][:, lo:hi].contiguous() for k_ in ("q", "k", "v", "g", "beta")}
        parts.append(gdn.gdn_varlen_fwd(cu_seqlens(lens).cuda(), sub["q"], sub["k"], sub["v"],
                                        sub["g"], sub["beta"])[0])
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(parts, dim=1), o)


def test_fp32_workload_sizes_on_simt_path():
    """The tiny fp32 workload runs the SIMT kernels; the bf16 workloads the tensor-core ones."""
    w0, w2 = workload(0), workload(2)
    s0 = gdn.gdn_shape(w0.B, w0.T, w0.H, w0.dk, w0.dv, 0)
    s2 = gdn.gdn_shape(w2.B, w2.T, w2.H, w2.dk, w2.dv, 1)
    lib = gdn.load()
    import ctypes
    assert lib.gdn_path(ctypes.byref(s0)) == 1
    assert lib.gdn_path(ctypes.byref(s2)) == 2


def test_benchmark_step_kept_products():
    """The benchmark's own step (bench.Runner: 8 chained 32768-token chunks,
    forward keeping its products, backward reading them) on the 256K-token
    workload: sampled heads against the oracle, and every output bitwise equal
    to the recomputing pair."""
    import bench

    w = workload(2)
    dev = torch.device("cuda", 0)
    kept = bench.Runner(w, dev, reuse=True)
    kept.step()
    torch.cuda.synchronize()
    grads = (kept.dq, kept.dk, kept.dv, kept.dg, kept.db, kept.dS[0])
    check_heads(w, kept.x, kept.o, kept.S[-1], grads, [0, 9])
    outs = [t.clone() for t in (kept.o, kept.S[-1]) + grads]
    del kept
    torch.cuda.empty_cache()
    rec = bench.Runner(w, dev, reuse=False)
    rec.step()
    torch.cuda.synchronize()
    for a, b in zip(outs, (rec.o, rec.S[-1], rec.dq, rec.dk, rec.dv, rec.dg, rec.db, rec.dS[0])):
        assert torch.equal(a, b)


def test_benchmark_short_conv_full_size():
    """The benchmark's short convolution (C = 6144, W = 4, SiLU, 256K tokens in
    8 chained chunks) on sampled channels against the oracle; the chained
    forward equals one call over the whole sequence."""
    from chunked_linear_recurrence_gated_gb300.inputs import CONV_BENCH, make_conv_inputs
    from oracle import short_conv as sc

    cfg = CONV_BENCH
    B, T, C, W = cfg["B"], cfg["T"], cfg["C"], cfg["W"]
    d = make_conv_inputs(B, T, C, W, dtype=BF, device="cuda", with_state=False)
    bounds = np.concatenate([[0], np.cumsum(cfg["chunks"])]).astype(int)
    n = len(cfg["chunks"])
    ys, states, s = [], [None], None
    for i in range(n):
        y, s = gdn.gdn_conv_fwd(d["x"][:, bounds[i]:bounds[i + 1]], d["w"], d["b"], s, "silu")
        ys.append(y)
        states.append(s)
    dxs, dw, db, ds = [None] * n, 0, 0, None
    for i in reversed(range(n)):
        sl = slice(bounds[i], bounds[i + 1])
        dx, dwi, dbi, ds = gdn.gdn_conv_bwd(d["x"][:, sl], d["w"], d["b"], states[i],
                                            d["dy"][:, sl], ds, "silu")
        dxs[i] = dx
        dw, db = dw + dwi, db + dbi
    y_full, _ = gdn.gdn_conv_fwd(d["x"], d["w"], d["b"], None, "silu")
    torch.cuda.synchronize()
    y = torch.cat(ys, dim=1)
    assert torch.equal(y, y_full)
    cols = torch.arange(3, C, 389)
    f64 = lambda t: t.double().cpu().numpy()
    y_ref, _ = sc.conv_fwd(f64(d["x"][..., cols]), f64(d["w"][cols]), f64(d["b"][cols]), None)
    dx_ref, dw_ref, db_ref, _ = sc.conv_bwd(f64(d["x"][..., cols]), f64(d["w"][cols]),
                                            f64(d["b"][cols]), None, f64(d["dy"][..., cols]))
    assert rel_err(y[..., cols], y_ref) <= FWD_TOL[BF]
    assert rel_err(torch.cat(dxs, dim=1)[..., cols], dx_ref) <= BWD_TOL[BF]
    assert rel_err(dw[cols], dw_ref) <= BWD_TOL[BF]
    assert rel_err(db[cols], db_ref) <= BWD_TOL[BF]
