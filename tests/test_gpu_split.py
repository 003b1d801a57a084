"""The split forward (state-transition / dense-kernel overlap, the StateFlow
review's split fraction f): splitting a chunk's blocks into segments whose Pre
kernel runs beside the previous segment's state chain, and carrying 16 or 32
value columns per chain CTA, must leave every result bit-identical to the
serial order. Also checked through the kept-products pair (the backward reads
what the split forward kept)."""
import pytest
import torch

from chunked_linear_recurrence_gated_gb300 import gdn
from chunked_linear_recurrence_gated_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

SETTINGS = [(1, 0, 2), (2, 0, 1), (2, 0, 2), (2, 300, 2), (2, 900, 2), (3, 0, 2), (4, 0, 2),
            (8, 0, 1), (16, 0, 2)]


@pytest.fixture(autouse=True)
def _restore_default_split():
    yield
    gdn.set_fwd_split(0, 0, 0)


def forward(d, saved=False):
    if saved:
        o, S, sv = gdn.gdn_chunk_fwd_save(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"])
        return o, S, sv
    return gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"])


@pytest.mark.parametrize("B,T,H", [(1, 64 * 37 + 11, 4), (2, 64 * 20, 3)])
def test_split_forward_bit_identical(B, T, H):
    x = make_inputs(B, T, H, 128, 128, dtype=torch.bfloat16, seed=B * 100 + H, decay="weak",
                    with_state=True)
    d = {k: v.cuda() for k, v in x.items()}
    gdn.set_fwd_split(1, 0, 1)
    o0, S0 = forward(d)
    torch.cuda.synchronize()
    for seg, pm, rg in SETTINGS:
        gdn.set_fwd_split(seg, pm, rg)
        o, S = forward(d)
        torch.cuda.synchronize()
        assert torch.equal(o, o0), (seg, pm, rg)
        assert torch.equal(S, S0), (seg, pm, rg)


def test_split_forward_kept_products_backward():
    x = make_inputs(1, 64 * 29, 2, 128, 128, dtype=torch.bfloat16, seed=3, decay="weak",
                    with_state=True)
    d = {k: v.cuda() for k, v in x.items()}
    gdn.set_fwd_split(1, 0, 1)
    o0, S0, sv0 = forward(d, saved=True)
    g0 = gdn.gdn_chunk_bwd_saved(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"], d["do"], sv0,
                                 dS_out=d["dS_out"])
    torch.cuda.synchronize()
    for seg, pm, rg in [(4, 0, 2), (2, 700, 1)]:
        gdn.set_fwd_split(seg, pm, rg)
        o, S, sv = forward(d, saved=True)
        g = gdn.gdn_chunk_bwd_saved(d["q"], d["k"], d["v"], d["g"], d["beta"], d["S_in"], d["do"],
                                    sv, dS_out=d["dS_out"])
        torch.cuda.synchronize()
        assert torch.equal(o, o0) and torch.equal(S, S0)
        for a, b in zip(g, g0):
            assert torch.equal(a, b)
