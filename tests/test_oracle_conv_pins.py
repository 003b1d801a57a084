"""Pins of the short-convolution oracle (oracle/short_conv.py) to things other
than itself: a library FIR filter, the SiLU of a library sigmoid, the
identity kernel, chunk chaining of the definition, and central finite
differences of every input of the backward."""
import numpy as np
import pytest
from scipy.signal import lfilter
from scipy.special import expit

from oracle import short_conv as sc


def rand(rng, *shape):
    return rng.standard_normal(shape)


def test_matches_library_fir_filter():
    """Zero incoming state: y[t, c] = sum_k h[k] x[t - k, c] with taps h[k] = w[c, W-1-k]."""
    rng = np.random.default_rng(0)
    B, T, C, W = 2, 37, 5, 4
    x, w, b = rand(rng, B, T, C), rand(rng, C, W), rand(rng, C)
    y, _ = sc.conv_fwd(x, w, b, None, act="none")
    for bb in range(B):
        for c in range(C):
            ref = lfilter(w[c, ::-1], [1.0], x[bb, :, c]) + b[c]
            np.testing.assert_allclose(y[bb, :, c], ref, rtol=0, atol=1e-12)


def test_incoming_state_is_the_preceding_inputs():
    """A nonzero state equals prepending those inputs and dropping their outputs."""
    rng = np.random.default_rng(1)
    B, T, C, W = 1, 20, 3, 4
    x, w = rand(rng, B, T, C), rand(rng, C, W)
    s = rand(rng, B, W - 1, C)
    y, _ = sc.conv_fwd(x, w, None, s, act="none")
    full = np.concatenate([s, x], axis=1)
    for c in range(C):
        ref = lfilter(w[c, ::-1], [1.0], full[0, :, c])[W - 1:]
        np.testing.assert_allclose(y[0, :, c], ref, rtol=0, atol=1e-12)


def test_silu_is_z_times_library_sigmoid():
    rng = np.random.default_rng(2)
    x, w, b = rand(rng, 1, 16, 4), rand(rng, 4, 3), rand(rng, 4)
    z, _ = sc.conv_fwd(x, w, b, None, act="none")
    y, _ = sc.conv_fwd(x, w, b, None, act="silu")
    np.testing.assert_allclose(y, z * expit(z), rtol=1e-13, atol=1e-15)


def test_identity_kernel_and_state_out():
    rng = np.random.default_rng(3)
    B, T, C, W = 2, 9, 3, 4
    x = rand(rng, B, T, C)
    w = np.zeros((C, W))
    w[:, W - 1] = 1.0  # the current token only
    s = rand(rng, B, W - 1, C)
    y, so = sc.conv_fwd(x, w, None, s, act="none")
    assert np.array_equal(y, x)
    assert np.array_equal(so, x[:, T - (W - 1):, :])
    # a chunk shorter than the state keeps part of the incoming state
    y2, so2 = sc.conv_fwd(x[:, :2], w, None, s, act="none")
    assert np.array_equal(so2, np.concatenate([s[:, 2:], x[:, :2]], axis=1))


@pytest.mark.parametrize("act", ["none", "silu"])
def test_chunk_chaining_is_exact(act):
    rng = np.random.default_rng(4)
    B, T, C, W = 2, 23, 4, 4
    x, w, b, dy = rand(rng, B, T, C), rand(rng, C, W), rand(rng, C), rand(rng, B, T, C)
    s0 = rand(rng, B, W - 1, C)
    y, s_end = sc.conv_fwd(x, w, b, s0, act)
    dx, dw, db, ds0 = sc.conv_bwd(x, w, b, s0, dy, None, act)
    cuts = [0, 2, 11, 23]  # includes a chunk shorter than W - 1
    ys, states, s = [], [s0], s0
    for a, e in zip(cuts[:-1], cuts[1:]):
        yi, s = sc.conv_fwd(x[:, a:e], w, b, s, act)
        ys.append(yi)
        states.append(s)
    assert np.array_equal(np.concatenate(ys, axis=1), y)
    assert np.array_equal(s, s_end)
    dxs, dws, dbs, ds = [None] * 3, [], [], None
    for i in reversed(range(3)):
        a, e = cuts[i], cuts[i + 1]
        dxi, dwi, dbi, ds = sc.conv_bwd(x[:, a:e], w, b, states[i], dy[:, a:e], ds, act)
        dxs[i] = dxi
        dws.append(dwi)
        dbs.append(dbi)
    np.testing.assert_allclose(np.concatenate(dxs, axis=1), dx, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ds, ds0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(sum(dws), dw, rtol=0, atol=1e-11)
    np.testing.assert_allclose(sum(dbs), db, rtol=0, atol=1e-11)


@pytest.mark.parametrize("T", [2, 7])
@pytest.mark.parametrize("act", ["none", "silu"])
def test_backward_against_finite_differences(T, act):
    rng = np.random.default_rng(5 + T)
    B, C, W = 2, 3, 4
    x, w, b = rand(rng, B, T, C), rand(rng, C, W), rand(rng, C)
    s = rand(rng, B, W - 1, C)
    dy, dso = rand(rng, B, T, C), rand(rng, B, W - 1, C)

    def loss(x_, w_, b_, s_):
        y, so = sc.conv_fwd(x_, w_, b_, s_, act)
        return float((y * dy).sum() + (so * dso).sum())

    dx, dw, db, ds = sc.conv_bwd(x, w, b, s, dy, dso, act)
    h = 1e-6
    for arr, grad, name in ((x, dx, "x"), (w, dw, "w"), (b, db, "b"), (s, ds, "state_in")):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + h
            lp = loss(x, w, b, s)
            arr[idx] = old - h
            lm = loss(x, w, b, s)
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-7, err_msg=name)
