"""GPU parity of the causal short convolution with carried boundary state
(include/gdn_conv.h) against the fp64 oracle, chunk chaining, edge cases and
determinism, through the C ABI."""
import numpy as np
import pytest
import torch

from chunked_linear_recurrence_gated_gb300 import gdn
from chunked_linear_recurrence_gated_gb300.inputs import make_conv_inputs
from helpers import BWD_TOL, FWD_TOL, np64, rel_err
from oracle import short_conv as sc

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def to_cuda(d):
    return {k: (v.cuda() if v is not None else None) for k, v in d.items()}


def oracle_of(d, act):
    x, w, b, s = np64(d["x"]), np64(d["w"]), None if d["b"] is None else np64(d["b"]), None
    if d["state_in"] is not None:
        s = np64(d["state_in"])
    y, so = sc.conv_fwd(x, w, b, s, act)
    dso = None if d["dstate_out"] is None else np64(d["dstate_out"])
    dx, dw, db, ds = sc.conv_bwd(x, w, b, s, np64(d["dy"]), dso, act)
    return y, so, dx, dw, db, ds


def run_gpu(d, act):
    y, so = gdn.gdn_conv_fwd(d["x"], d["w"], d["b"], d["state_in"], act)
    dx, dw, db, ds = gdn.gdn_conv_bwd(d["x"], d["w"], d["b"], d["state_in"], d["dy"],
                                      d["dstate_out"], act)
    torch.cuda.synchronize()
    return y, so, dx, dw, db, ds


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("W", [2, 4, 8])
@pytest.mark.parametrize("act", ["none", "silu"])
def test_conv_parity(dtype, W, act):
    # 300 tokens: several forward tiles (64) and backward tiles (256) plus a ragged tail
    d = make_conv_inputs(2, 300, 40, W, dtype=DT[dtype], seed=W + len(act))
    ref = oracle_of(d, act)
    got = run_gpu(to_cuda(d), act)
    names = ["y", "state_out", "dx", "dw", "db", "dstate_in"]
    for name, g, r in zip(names, got, ref):
        tol = FWD_TOL[DT[dtype]] if name in ("y", "state_out") else BWD_TOL[DT[dtype]]
        assert rel_err(g, r) <= tol, (name, rel_err(g, r))
    # the outgoing state is a copy of inputs: exact
    assert np.array_equal(np64(got[1]), ref[1])


@pytest.mark.parametrize("T", [0, 1, 2, 3, 65, 256, 257])
def test_conv_edge_lengths(T):
    d = make_conv_inputs(1, T, 16, 4, dtype=torch.float32, seed=T)
    ref = oracle_of(d, "silu")
    got = run_gpu(to_cuda(d), "silu")
    for name, g, r in zip(["y", "state_out", "dx", "dw", "db", "dstate_in"], got, ref):
        if np.asarray(r).size:
            assert rel_err(g, r) <= 1e-5, (T, name, rel_err(g, r))
    if T == 0:
        assert torch.equal(got[1].cpu(), d["state_in"])
        assert torch.equal(got[5].cpu(), d["dstate_out"])


def test_conv_zero_state_and_no_bias():
    d = make_conv_inputs(2, 130, 24, 4, dtype=torch.float32, seed=9, with_state=False,
                         with_bias=False)
    ref = oracle_of(d, "none")
    got = run_gpu(to_cuda(d), "none")
    for name, g, r in zip(["y", "state_out", "dx", "dw"], got[:4], ref[:4]):
        assert rel_err(g, r) <= 1e-5, name
    assert got[4] is None


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_chunk_chaining(dtype):
    """8 chained chunks vs one call: y and the states bit-identical; dx, dw, db
    equal up to the summation order of the W - 1 tokens at each boundary."""
    d = to_cuda(make_conv_inputs(1, 600, 64, 4, dtype=DT[dtype], seed=3))
    full = run_gpu(d, "silu")
    cuts = [0, 2, 64, 100, 256, 257, 400, 599, 600]
    ys, states, s = [], [d["state_in"]], d["state_in"]
    for a, e in zip(cuts[:-1], cuts[1:]):
        y, s = gdn.gdn_conv_fwd(d["x"][:, a:e].contiguous(), d["w"], d["b"], s, "silu")
        ys.append(y)
        states.append(s)
    assert torch.equal(torch.cat(ys, dim=1), full[0])
    assert torch.equal(s, full[1])
    dxs, dws, dbs, ds = [None] * (len(cuts) - 1), [], [], d["dstate_out"]
    for i in reversed(range(len(cuts) - 1)):
        a, e = cuts[i], cuts[i + 1]
        dx, dw, db, ds = gdn.gdn_conv_bwd(d["x"][:, a:e].contiguous(), d["w"], d["b"], states[i],
                                          d["dy"][:, a:e].contiguous(), ds, "silu")
        dxs[i] = dx
        dws.append(dw)
        dbs.append(db)
    torch.cuda.synchronize()
    tol = 1e-5 if dtype == "f32" else 1e-2
    assert rel_err(torch.cat(dxs, dim=1), full[2]) <= tol
    assert rel_err(ds, full[5]) <= tol
    assert rel_err(sum(dws), full[3]) <= 1e-5
    assert rel_err(sum(dbs), full[4]) <= 1e-5


def test_conv_deterministic_and_wide():
    """The benchmark's channel count (16 heads x 384) on a short sequence; two
    runs bitwise equal; sampled outputs against the oracle."""
    d = to_cuda(make_conv_inputs(1, 700, 16 * 384, 4, dtype=torch.bfloat16, seed=11))
    a = run_gpu(d, "silu")
    b = run_gpu(d, "silu")
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    cols = torch.arange(0, 16 * 384, 97)
    sub = {k: (v[..., cols].cpu() if k != "w" and k != "b" and v is not None else v)
           for k, v in d.items()}
    sub["w"] = d["w"][cols].cpu()
    sub["b"] = d["b"][cols].cpu()
    ref = oracle_of(sub, "silu")
    got = [a[0][..., cols], a[1][..., cols], a[2][..., cols], a[3][cols], a[4][cols],
           a[5][..., cols]]
    for name, g, r in zip(["y", "state_out", "dx", "dw", "db", "dstate_in"], got, ref):
        tol = 2e-2 if name in ("y", "state_out") else 3e-2
        assert rel_err(g, r) <= tol, name
