"""Pins of the oracle's projection (the x_proj and dt_proj nodes of the "Mamba 模型"
block flowchart) to things other than itself: the product written out as
explicit sums, row selection by one-hot weights (catches a transposed operand
or swapped batch/row index), the x_proj -> dt_proj chain against the product
of the weights (associativity), and the softplus epilogue against the
definition log(1 + e^v)."""
import numpy as np

import oracle


def test_projection_is_the_explicit_sum():
    rng = np.random.default_rng(0)
    W = rng.normal(size=(5, 7))
    X = rng.normal(size=(3, 7, 4))
    b = rng.normal(size=5)
    got = oracle.proj(W, X, bias=b)
    ref = np.zeros((3, 5, 4))
    for bb in range(3):
        for m in range(5):
            for n in range(4):
                s = b[m]
                for k in range(7):
                    s += W[m, k] * X[bb, k, n]
                ref[bb, m, n] = s
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_one_hot_rows_select_input_rows():
    rng = np.random.default_rng(1)
    X = rng.normal(size=(2, 6, 9))
    perm = [4, 0, 5, 2]
    W = np.zeros((4, 6))
    W[np.arange(4), perm] = 1.0
    assert np.array_equal(oracle.proj(W, X), X[:, perm, :])


def test_x_proj_then_dt_proj_is_the_weight_product():
    rng = np.random.default_rng(2)
    D, R, N, L = 12, 3, 2, 10
    Wx = rng.normal(size=(R + 2 * N, D))
    Wdt = rng.normal(size=(D, R))
    X = rng.normal(size=(2, D, L))
    x_dbl = oracle.proj(Wx, X)
    delta = oracle.proj(Wdt, x_dbl[:, :R])
    assert np.allclose(delta, oracle.proj(Wdt @ Wx[:R], X), rtol=1e-12, atol=1e-12)


def test_softplus_epilogue():
    v = np.linspace(-30.0, 30.0, 61)
    W = np.eye(61)
    got = oracle.proj(W, v.reshape(1, 61, 1), softplus=True)[0, :, 0]
    assert np.allclose(got, np.logaddexp(0.0, v), rtol=1e-14, atol=0)
