"""gdn_chunk_fwd_noalloc: the chunk forward for callers that cannot allocate
device memory (its scratch is a fixed array inside the library). Checked
through the C ABI against gdn_chunk_fwd with a caller-provided workspace, on
two calls in a row (the second reuses the array the first one left behind).

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import pytest
import torch

from chunked_linear_recurrence_gated_gb300 import gdn
from chunked_linear_recurrence_gated_gb300.inputs import make_inputs
from helpers import FWD_TOL, rel_err

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_noalloc(d, S_in):
    lib = gdn.load()
    q = d["q"]
    B, T, H, dk = q.shape
    dv = d["v"].shape[-1]
    o = torch.full((B, T, H, dv), float("nan"), dtype=q.dtype, device=q.device)
    S_out = torch.full((B, H, dk, dv), float("nan"), dtype=torch.float32, device=q.device)
    shape = gdn.shape_of(q, d["v"])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.gdn_chunk_fwd_noalloc(ctypes.byref(shape), _ptr(q), _ptr(d["k"]), _ptr(d["v"]),
                                   _ptr(d["g"]), _ptr(d["beta"]), _ptr(S_in), _ptr(o),
                                   _ptr(S_out), stream)
    return rc, o, S_out


@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 128, 128), (torch.float32, 64, 64)])
def test_noalloc_matches_workspace_call_twice(dtype, dk, dv):
    for seed in (31, 32):  # two calls in a row, different inputs
        x = make_inputs(2, 333, 3, dk, dv, dtype=dtype, seed=seed, decay="weak",
                        with_state=True)
        d = {k: v.cuda() for k, v in x.items()}
        o_ref, S_ref = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"])
        rc, o, S_out = call_noalloc(d, d["S_in"])
        torch.cuda.synchronize()
        assert rc == 0, gdn.gdn_status_str(rc)
        assert rel_err(o, o_ref) <= FWD_TOL[dtype]
        assert rel_err(S_out, S_ref) <= FWD_TOL[dtype]
        # same kernels, same arithmetic: the results are in fact identical
        assert torch.equal(o, o_ref) and torch.equal(S_out, S_ref)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = gdn.load()
    shape = gdn.gdn_shape(1, 1 << 20, 16, 128, 128, 1)  # needs far more than 64 MiB
    assert lib.gdn_chunk_workspace_bytes(ctypes.byref(shape), 0) > (64 << 20)
    fake = ctypes.c_void_p(1 << 20)
    rc = lib.gdn_chunk_fwd_noalloc(ctypes.byref(shape), *([fake] * 5), None, fake, None, None)
    assert rc == 3  # GDN_ERR_WORKSPACE, nothing launched
    bad = gdn.gdn_shape(1, 64, 2, 96, 128, 1)
    rc = lib.gdn_chunk_fwd_noalloc(ctypes.byref(bad), *([fake] * 5), None, fake, None, None)
    assert rc == 2  # GDN_ERR_UNSUPPORTED, as gdn_chunk_fwd reports it


def test_noalloc_status_reports_a_timeout_and_resets():
    """The no-allocation forward's device status (a bounded wait that gave up)
    is readable without a workspace pointer: the bounded-wait self-check on the
    scratch's status word reports GDN_ERR_TIMEOUT through gdn_noalloc_status,
    reading resets it, and the next call still computes correctly."""
    assert gdn.gdn_noalloc_status() == 0
    assert gdn.diag_wait_timeout_noalloc(limit_log2=20) == 0
    assert gdn.gdn_noalloc_status() == 5  # GDN_ERR_TIMEOUT
    assert gdn.gdn_noalloc_status() == 0
    x = make_inputs(1, 200, 2, 128, 128, dtype=torch.bfloat16, seed=33, decay="weak",
                    with_state=True)
    d = {k: v.cuda() for k, v in x.items()}
    o_ref, S_ref = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"])
    rc, o, S_out = call_noalloc(d, d["S_in"])
    assert rc == 0
    assert gdn.gdn_noalloc_status() == 0
    assert torch.equal(o, o_ref) and torch.equal(S_out, S_ref)
