"""Pins of the fp64 CPU oracle to mathematics, not to itself.

Each test fixes a result the oracle must reproduce from something outside its
own loop: a hand-worked example, the explicit product of transition matrices,
closed forms for beta = 0 and for the ungated delta rule with orthonormal keys,
the write invariant S_t k_t = v_t, central finite differences, and the
64-token chunkwise (WY) formulation derived separately.
"""
import os

import numpy as np
import pytest

import oracle
from oracle import wy

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(7)


def rand_problem(B=1, T=6, H=1, dk=5, dv=3, decay="default", seed=0, unit_keys=True):
    r = np.random.default_rng(seed)
    q = r.normal(size=(B, T, H, dk))
    k = r.normal(size=(B, T, H, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = r.normal(size=(B, T, H, dv))
    beta = 1 / (1 + np.exp(-r.normal(size=(B, T, H))))
    z = r.normal(size=(B, T, H))
    if decay == "default":
        g = -np.log1p(np.exp(z + 2))
    elif decay == "weak":
        g = -0.1 * np.log1p(np.exp(z - 5))
    else:
        g = np.zeros_like(z)
    S_in = r.normal(size=(B, H, dk, dv)) * 0.5
    return q, k, v, g, beta, S_in


# ---------------------------------------------------------------- forward pins

def test_scalar_worked_example():
    rows = []
    with open(os.path.join(GOLDEN, "scalar_worked_example.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            if parts[0] == "S0":
                S0 = float(parts[1])
            else:
                rows.append([float(x) for x in parts])
    rows = np.array(rows)
    T = len(rows)
    alpha, beta, k, v, q, o_ref, S_ref = (rows[:, i] for i in range(1, 8))
    sh = (1, T, 1, 1)
    o, S_out = oracle.fwd(q.reshape(sh), k.reshape(sh), v.reshape(sh),
                          np.log(alpha).reshape(1, T, 1), beta.reshape(1, T, 1),
                          np.array([[[[S0]]]]))
    np.testing.assert_allclose(o.ravel(), o_ref, rtol=0, atol=1e-15)
    assert abs(S_out.ravel()[0] - S_ref[-1]) < 1e-15
    # every prefix ends in the tabulated state
    for t in range(1, T + 1):
        _, St = oracle.fwd(q.reshape(sh)[:, :t], k.reshape(sh)[:, :t], v.reshape(sh)[:, :t],
                           np.log(alpha).reshape(1, T, 1)[:, :t],
                           beta.reshape(1, T, 1)[:, :t], np.array([[[[S0]]]]))
        assert abs(St.ravel()[0] - S_ref[t - 1]) < 1e-15


def brute_force(q, k, v, g, beta, S_in):
    """Explicit unrolled sum of products of the d_k x d_k transition matrices.

    S_t = S_0 P(1..t) + sum_s beta_s v_s k_s^T P(s+1..t),
    P(a..b) = A_a A_{a+1} ... A_b,  A_s = alpha_s (I - beta_s k_s k_s^T).
    No recurrence is stepped: each S_t is formed from scratch.
    """
    T, dk = k.shape
    dv = v.shape[1]
    A = [np.exp(g[s]) * (np.eye(dk) - beta[s] * np.outer(k[s], k[s])) for s in range(T)]

    def P(a, b):
        out = np.eye(dk)
        for s in range(a, b + 1):
            out = out @ A[s]
        return out

    S0 = S_in.T  # recurrence orientation: d_v x d_k
    o = np.zeros((T, dv))
    St = None
    for t in range(T):
        St = S0 @ P(0, t)
        for s in range(t + 1):
            St = St + beta[s] * np.outer(v[s], k[s]) @ P(s + 1, t)
        o[t] = St @ q[t]
    return o, St.T


@pytest.mark.parametrize("decay", ["default", "weak", "zero"])
@pytest.mark.parametrize("dims", [(5, 3), (3, 7), (8, 8)])
def test_forward_matches_brute_force(decay, dims):
    dk, dv = dims
    q, k, v, g, beta, S_in = rand_problem(T=7, dk=dk, dv=dv, decay=decay, seed=dk * 10 + dv,
                                          unit_keys=False)
    o, S_out = oracle.fwd(q, k, v, g, beta, S_in)
    o_ref, S_ref = brute_force(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0],
                               S_in[0, 0])
    np.testing.assert_allclose(o[0, :, 0], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S_out[0, 0], S_ref, rtol=0, atol=1e-12)


def test_beta_zero_closed_form():
    q, k, v, g, beta, S_in = rand_problem(B=2, T=40, H=3, dk=6, dv=4, seed=3)
    beta[:] = 0.0
    o, S_out = oracle.fwd(q, k, v, g, beta, S_in)
    gam = np.cumsum(g, axis=1)  # [B, T, H]
    # o_t = exp(gamma_t) S_in q_t  ->  with the stored state M = S^T: o_t = exp(gamma_t) M^T q_t
    o_ref = np.exp(gam)[..., None] * np.einsum("bthi,bhij->bthj", q, S_in)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S_out, np.exp(gam[:, -1])[..., None, None] * S_in,
                               rtol=1e-12, atol=1e-14)


def test_ungated_orthonormal_keys_store_values():
    """g = 0, beta = 1, keys = the standard basis: the state ends as exactly V."""
    d = 6
    T = d
    r = np.random.default_rng(11)
    basis = np.linalg.qr(r.normal(size=(d, d)))[0]  # orthonormal rows
    k = basis.reshape(1, T, 1, d)
    q = r.normal(size=(1, T, 1, d))
    v = r.normal(size=(1, T, 1, 4))
    g = np.zeros((1, T, 1))
    beta = np.ones((1, T, 1))
    S_in = r.normal(size=(1, 1, d, 4))
    _, S_out = oracle.fwd(q, k, v, g, beta, S_in)
    # S_T k_j = v_j for every key: with M = S^T this is M^T k_j = v_j.
    for j in range(T):
        np.testing.assert_allclose(S_out[0, 0].T @ basis[j], v[0, j, 0], atol=1e-12)


@pytest.mark.parametrize("decay", ["default", "weak"])
def test_write_invariant(decay):
    """beta = 1 and |k| = 1 give S_t k_t = v_t, so querying with q_t = k_t returns v_t."""
    q, k, v, g, beta, S_in = rand_problem(B=1, T=50, H=2, dk=8, dv=5, decay=decay, seed=5)
    beta[:] = 1.0
    o, _ = oracle.fwd(k, k, v, g, beta, S_in)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_chunkwise_wy_matches_token_loop(T):
    q, k, v, g, beta, S_in = rand_problem(B=2, T=T, H=2, dk=16, dv=12, seed=T, decay="weak")
    o, S_out = oracle.fwd(q, k, v, g, beta, S_in)
    o2, S2 = wy.fwd(q, k, v, g, beta, S_in)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-11 * max(1, np.abs(o).max()))
    np.testing.assert_allclose(S2, S_out, rtol=0, atol=1e-11 * max(1, np.abs(S_out).max()))


def test_chaining_is_bitwise_forward():
    q, k, v, g, beta, S_in = rand_problem(B=1, T=300, H=2, dk=8, dv=6, seed=21)
    o, S_out = oracle.fwd(q, k, v, g, beta, S_in)
    cut = [0, 64, 128, 300]
    S = S_in
    parts = []
    for a, b in zip(cut[:-1], cut[1:]):
        oc, S = oracle.fwd(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b], S)
        parts.append(oc)
    assert np.array_equal(np.concatenate(parts, axis=1), o)
    assert np.array_equal(S, S_out)


def test_varlen_equals_separate_sequences():
    lens = [5, 64, 1, 90]
    T = sum(lens)
    q, k, v, g, beta, _ = rand_problem(B=1, T=T, H=2, dk=8, dv=4, seed=9)
    S0 = np.random.default_rng(1).normal(size=(len(lens), 2, 8, 4))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o, Sf = oracle.varlen_fwd(cu, q, k, v, g, beta, S0)
    for s in range(len(lens)):
        a, b = cu[s], cu[s + 1]
        os_, Ss = oracle.fwd(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b],
                             S0[s:s + 1])
        assert np.array_equal(o[:, a:b], os_)
        assert np.array_equal(Sf[s], Ss[0])


def test_invalid_arguments_raise():
    q, k, v, g, beta, S_in = rand_problem()
    with pytest.raises(ValueError):
        oracle.varlen_fwd(np.array([0, 4, 3, 6], np.int32), q, k, v, g, beta)
    with pytest.raises(ValueError):
        oracle.varlen_fwd(np.array([1, 6], np.int32), q, k, v, g, beta)


# --------------------------------------------------------------- backward pins

def loss(q, k, v, g, beta, S_in, dout, dS_out):
    o, S_out = oracle.fwd(q, k, v, g, beta, S_in, nthreads=1)
    return float(np.sum(o * dout) + np.sum(S_out * dS_out))


@pytest.mark.parametrize("decay", ["default", "weak"])
@pytest.mark.parametrize("T", [7, 70])
def test_backward_matches_finite_differences(decay, T):
    dk, dv = 4, 3
    q, k, v, g, beta, S_in = rand_problem(T=T, dk=dk, dv=dv, decay=decay, seed=T + 100,
                                          unit_keys=False)
    r = np.random.default_rng(T)
    dout = r.normal(size=(1, T, 1, dv))
    dS_out = r.normal(size=(1, 1, dk, dv))
    grads = oracle.bwd(q, k, v, g, beta, S_in, dout, dS_out)
    args = [q, k, v, g, beta, S_in]
    names = ["q", "k", "v", "g", "beta", "S_in"]
    h = 1e-6
    for ai, (name, grad) in enumerate(zip(names, grads)):
        x = args[ai]
        flat = x.reshape(-1)
        idx = np.arange(flat.size) if flat.size <= 40 else r.choice(flat.size, 40, replace=False)
        for i in idx:
            orig = flat[i]
            flat[i] = orig + h
            lp = loss(*args, dout, dS_out)
            flat[i] = orig - h
            lm = loss(*args, dout, dS_out)
            flat[i] = orig
            fd = (lp - lm) / (2 * h)
            an = grad.reshape(-1)[i]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, i, fd, an)


def test_backward_beta_zero_closed_form():
    B, T, H, dk, dv = 1, 30, 2, 5, 4
    q, k, v, g, beta, S_in = rand_problem(B=B, T=T, H=H, dk=dk, dv=dv, seed=33)
    beta[:] = 0.0
    r = np.random.default_rng(2)
    dout = r.normal(size=(B, T, H, dv))
    dS_out = r.normal(size=(B, H, dk, dv))
    dq, dk_, dv_, dg, dbeta, dS_in = oracle.bwd(q, k, v, g, beta, S_in, dout, dS_out)
    gam = np.cumsum(g, axis=1)
    E = np.exp(gam)  # [B, T, H]
    # o_t = e^{gamma_t} M^T q_t
    np.testing.assert_allclose(dq, E[..., None] * np.einsum("bhij,bthj->bthi", S_in, dout),
                               rtol=1e-11, atol=1e-13)
    assert np.abs(dv_).max() == 0.0
    assert np.abs(dk_).max() == 0.0
    ref_dS = np.einsum("bth,bthi,bthj->bhij", E, q, dout) + E[:, -1][..., None, None] * dS_out
    np.testing.assert_allclose(dS_in, ref_dS, rtol=1e-11, atol=1e-13)
    # dgamma_t = e^{gamma_t} do_t . (M^T q_t); the end term is e^{gamma_T} <dS_out, M>
    dgam = E * np.einsum("bthj,bthi,bhij->bth", dout, q, S_in)
    dgam[:, -1] += E[:, -1] * np.einsum("bhij,bhij->bh", dS_out, S_in)
    dg_ref = np.flip(np.cumsum(np.flip(dgam, 1), 1), 1)
    np.testing.assert_allclose(dg, dg_ref, rtol=1e-11, atol=1e-13)
    # beta = 0 does not make dbeta vanish: it is k_t^T D_t e_t
    assert np.abs(dbeta).max() > 1e-3


def test_chaining_is_bitwise_backward():
    q, k, v, g, beta, S_in = rand_problem(B=1, T=200, H=2, dk=8, dv=6, seed=44, decay="weak")
    r = np.random.default_rng(4)
    dout = r.normal(size=(1, 200, 2, 6))
    dS_out = r.normal(size=(1, 2, 8, 6))
    full = oracle.bwd(q, k, v, g, beta, S_in, dout, dS_out)
    cut = [0, 128, 200]
    _, S_mid = oracle.fwd(q[:, :128], k[:, :128], v[:, :128], g[:, :128], beta[:, :128], S_in)
    second = oracle.bwd(q[:, 128:], k[:, 128:], v[:, 128:], g[:, 128:], beta[:, 128:], S_mid,
                        dout[:, 128:], dS_out)
    first = oracle.bwd(q[:, :128], k[:, :128], v[:, :128], g[:, :128], beta[:, :128], S_in,
                       dout[:, :128], second[5])
    for i in range(5):
        assert np.array_equal(np.concatenate([first[i], second[i]], axis=1), full[i])
    assert np.array_equal(first[5], full[5])
    del cut


@pytest.mark.parametrize("T", [1, 64, 130])
def test_chunkwise_wy_backward_matches_token_loop(T):
    q, k, v, g, beta, S_in = rand_problem(B=1, T=T, H=2, dk=16, dv=12, seed=T + 5,
                                          decay="weak")
    r = np.random.default_rng(T)
    dout = r.normal(size=(1, T, 2, 12))
    dS_out = r.normal(size=(1, 2, 16, 12))
    ref = oracle.bwd(q, k, v, g, beta, S_in, dout, dS_out)
    got = wy.bwd(q, k, v, g, beta, S_in, dout, dS_out)
    for name, a, b in zip(["dq", "dk", "dv", "dg", "dbeta", "dS_in"], got, ref):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-9 * max(1, np.abs(b).max()),
                                   err_msg=name)


def test_varlen_backward_equals_separate_sequences():
    lens = [64, 3, 100]
    T = sum(lens)
    q, k, v, g, beta, _ = rand_problem(B=1, T=T, H=2, dk=6, dv=5, seed=17)
    r = np.random.default_rng(3)
    S0 = r.normal(size=(3, 2, 6, 5))
    dSf = r.normal(size=(3, 2, 6, 5))
    dout = r.normal(size=(1, T, 2, 5))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    got = oracle.varlen_bwd(cu, q, k, v, g, beta, S0, dout, dSf)
    for s in range(3):
        a, b = cu[s], cu[s + 1]
        ref = oracle.bwd(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b], S0[s:s + 1],
                         dout[:, a:b], dSf[s:s + 1])
        for i in range(5):
            assert np.array_equal(got[i][:, a:b], ref[i])
        assert np.array_equal(got[5][s], ref[5][0])
