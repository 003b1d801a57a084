"""Host-side logic: chunk partition (hybrid alpha family) and workload recipe."""
import numpy as np

from chunked_linear_recurrence_gated_gb300.inputs import (cu_seqlens, make_inputs,
                                                          varlen_lengths, workloads)
from chunked_linear_recurrence_gated_gb300.partition import hybrid_boundaries


def test_hybrid_partition_alpha_half():
    # a = L_lin C_lin + C_dense = 4, b = 1: f(x) = 4x + x^2/2; boundaries blend
    # i*T/N with the equal-cost offsets, rounded half-up to 64.
    b = hybrid_boundaries(131072, 8, 0.5)
    assert b == [0, 31360, 49152, 64704, 79104, 92800, 105920, 118656, 131072]


def test_hybrid_partition_limits():
    T, N = 65536, 4
    assert hybrid_boundaries(T, N, 0.0) == [0, 16384, 32768, 49152, 65536]
    b1 = hybrid_boundaries(T, N, 1.0)
    f = lambda x: 4 * x + x * x / 2
    costs = [f(b1[i + 1]) - f(b1[i]) for i in range(N)]
    assert max(costs) / min(costs) < 1.01  # equal cost up to 64-rounding
    assert all(x % 64 == 0 for x in b1)


def test_varlen_lengths_recipe():
    L = varlen_lengths()
    assert sum(L) == 131072
    assert all(x % 64 == 0 and 64 <= x <= 65536 for x in L)
    cu = cu_seqlens(L).numpy()
    assert cu[0] == 0 and cu[-1] == 131072 and np.all(np.diff(cu) > 0)


def test_workloads_shapes():
    ws = workloads()
    assert [sum(w.chunks) for w in ws[:4]] == [w.T for w in ws[:4]]
    assert all(c % 64 == 0 for w in ws[:4] for c in w.chunks)


def test_inputs_seeded_and_normalised():
    a = make_inputs(1, 70, 2, 16, 8, seed=5)
    b = make_inputs(1, 70, 2, 16, 8, seed=5)
    for key in a:
        assert a[key].equal(b[key])
    n = a["k"].float().norm(dim=-1)
    assert (n - 1).abs().max() < 1e-2
    assert (a["g"].float() < 0).all() and ((a["beta"].float() > 0) & (a["beta"].float() < 1)).all()


def test_bench_models_every_compute_kernel_the_library_marks():
    """Every compute kernel name the library's timing hook can report has a
    design-bytes / flops model in bench.py (the dominant-kernel roofline needs
    one), and the reference arm reports the GPU arm's workload config."""
    import glob
    import os
    import re

    import bench
    from chunked_linear_recurrence_gated_gb300.inputs import workload

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    names = set()
    for path in glob.glob(os.path.join(root, "chunked_linear_recurrence_gated_gb300", "csrc", "*.cu")):
        text = open(path).read()
        names |= set(re.findall(r'prof_mark\(st, "([a-z_0-9]+)"', text))
        names |= set(re.findall(r'"(tc_[a-z_]+)" : "(?:tc_[a-z_]+)"', text))
        names |= set(re.findall(r'"tc_[a-z_]+" : "(tc_[a-z_]+)"', text))
    helpers = {"status", "varlen_prep", "conv_fwd", "conv_bwd", "conv_reduce"}
    compute = sorted(names - helpers)
    assert "tc_grad" in compute and "tc_chain_fwd_keep" in compute and "tc_chain_fwd" in compute
    for name in compute:
        model = bench.kernel_model(name, 128, 128)
        assert model is not None and model[0] > 0, name
    # backward-phase kernels are credited with the backward's algorithmic bytes
    for name in compute:
        if "grad" in name or "rev" in name or "bwd" in name:
            assert bench.KERNEL_PHASE.get(name) == "bwd", name
    w = workload(bench.WORKLOAD_INDEX)
    cfg = bench.workload_config(w, 1, False)
    assert cfg["T"] == w.T and cfg["chunks"] == w.chunks and cfg["H"] == w.H


def test_bench_kernel_roofline_follows_the_survey_bytes():
    """The dominant kernel's roofline counts SURVEY 8(d)'s algorithmic bytes
    per token-head (fwd 4dk + 4dv + 4, bwd 8dk + 6dv + 8 at bf16) times the
    token-heads of its launches, over the summed launch time."""
    import bench
    from chunked_linear_recurrence_gated_gb300.inputs import workload

    w = workload(bench.WORKLOAD_INDEX)
    assert bench.alg_bytes_per_token_head(128, 128) == (1028, 1800)
    units = [32768 * 16] * 8
    r = bench.kernel_roofline("tc_grad", [0.5] * 8, units, w, 1000.0, "test")
    assert abs(r["achieved"] - 1800 * 32768 * 16 / 0.5e-3 / 1e9) < 1e-6
    assert abs(r["frac"] - r["achieved"] / 1000.0) < 1e-12
    r = bench.kernel_roofline("tc_pre", [0.5, 0.25], [100, 50], w, 1000.0, "test")
    assert abs(r["achieved"] - 1028 * 150 / 0.75e-3 / 1e9) < 1e-6
    # uneven launches: total units over total time, not the largest launch
    r2 = bench.kernel_roofline("tc_grad", [1.0, 0.1], [1000, 100], w, 1000.0, "test")
    assert abs(r2["achieved"] - 1800 * 1100 / 1.1e-3 / 1e9) < 1e-6
