"""Failure detection without a GPU fault: a kernel whose bounded wait runs out
(an mbarrier nothing arrives at) records GDN_ERR_TIMEOUT in the workspace's
status word and returns; the host reads it, and the context stays usable."""
import pytest
import torch

import oracle
from chunked_linear_recurrence_gated_gb300 import gdn
from chunked_linear_recurrence_gated_gb300.inputs import make_inputs
from helpers import FWD_TOL, rel_err, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    ws = gdn.alloc_workspace(4096, "cuda")
    assert gdn.diag_wait_timeout(ws, limit_log2=20) == 0
    assert gdn.gdn_workspace_status(ws) == 5  # GDN_ERR_TIMEOUT; reading resets the word
    assert gdn.gdn_workspace_status(ws) == 0
    # the same context keeps computing correctly
    x = make_inputs(1, 130, 2, 128, 128, dtype=torch.bfloat16, seed=21, with_state=True)
    d = to_dev(x)
    o, S = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"])
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S_in"])
    assert rel_err(o, o_ref) <= FWD_TOL[torch.bfloat16]
    assert rel_err(S, S_ref) <= FWD_TOL[torch.bfloat16]
