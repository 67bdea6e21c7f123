"""Pins for the SwiGLU part of the CPU oracle (the variant of the block on the
70B page, section "The MLP Block"), checked against closed forms, scipy's
logistic function, permutation weights that reduce the products to indexing,
central differences of the oracle's own forward, and the partition algebra
(sharded == unsharded).

A slip the pins catch: gate and up halves swapped (the permutation test gives
the halves different inputs and the gate a sign-sensitive Swish), Swish taken
as sigmoid or as x * sigmoid(-x) (closed forms), a wrong derivative (finite
differences and scipy), a shard gathering the wrong up columns (sharded ==
unsharded with t up to 6).
"""

import numpy as np
import pytest
from scipy.special import expit

import oracle


def rng(seed):
    return np.random.default_rng(seed)


def test_swish_special_values():
    # Swish(0) = 0, Swish'(0) = sigmoid(0) = 1/2
    assert oracle.swish(0.0) == 0.0
    assert abs(oracle.swish_grad(0.0) - 0.5) < 1e-15
    # far tails: Swish(x) -> x for x >> 0, -> 0 for x << 0
    assert abs(oracle.swish(40.0) - 40.0) < 1e-12
    assert abs(oracle.swish(-40.0)) < 1e-15
    assert oracle.swish(-800.0) == 0.0 or abs(oracle.swish(-800.0)) < 1e-300


@pytest.mark.parametrize("x", [-7.0, -2.0, -0.6, 0.2, 1.0, 3.5, 9.0])
def test_swish_is_x_times_logistic(x):
    assert abs(oracle.swish(x) - x * expit(x)) < 1e-14 * max(1.0, abs(x))


@pytest.mark.parametrize("x", [-3.0, -1.0, 0.4, 2.5])
def test_swish_odd_part_identity(x):
    # sigmoid(x) + sigmoid(-x) = 1  =>  Swish(x) - Swish(-x) = x
    assert abs(oracle.swish(x) - oracle.swish(-x) - x) < 1e-14 * max(1.0, abs(x))


@pytest.mark.parametrize("x", [-4.0, -1.2, 0.1, 0.9, 3.3])
def test_swish_grad_matches_central_difference_and_closed_form(x):
    e = 1e-5
    fd = (oracle.swish(x + e) - oracle.swish(x - e)) / (2 * e)
    assert abs(fd - oracle.swish_grad(x)) < 1e-9
    s = expit(x)
    assert abs(oracle.swish_grad(x) - (s + x * s * (1 - s))) < 1e-14


def test_swiglu_forward_with_permutation_weights():
    # gate column j reads input pg[j] scaled by dg[j]; up column j reads pu[j]
    T, h, f = 4, 5, 7
    r = rng(21)
    X = r.standard_normal((T, h))
    pg, pu = r.integers(0, h, size=f), r.integers(0, h, size=f)
    dg, du = r.uniform(0.5, 2.0, size=f), r.uniform(-2.0, -0.5, size=f)
    W1 = np.zeros((h, 2 * f))
    W1[pg, np.arange(f)] = dg
    W1[pu, f + np.arange(f)] = du
    b1 = r.standard_normal(2 * f)
    sigma = r.permutation(f)[:h]
    c = r.uniform(-2.0, 2.0, size=h)
    W2 = np.zeros((f, h))
    W2[sigma, np.arange(h)] = c
    b2 = r.standard_normal(h)
    out = oracle.swiglu_forward(X, W1, b1, W2, b2)
    G = dg[None, :] * X[:, pg] + b1[None, :f]
    Up = du[None, :] * X[:, pu] + b1[None, f:]
    Y = G * expit(G) * Up
    Z = c[None, :] * Y[:, sigma] + b2[None, :]
    np.testing.assert_allclose(out["GU"][:, :f], G, atol=1e-14)
    np.testing.assert_allclose(out["GU"][:, f:], Up, atol=1e-14)
    np.testing.assert_allclose(out["Y"], Y, atol=1e-13)
    np.testing.assert_allclose(out["Z"], Z, atol=1e-13)


def test_swiglu_constant_gate_reduces_to_linear():
    # W_gate = 0, b_gate = c: Y = Swish(c) (X W_up + b_up), a linear map
    T, h, f = 3, 4, 5
    r = rng(22)
    X = r.standard_normal((T, h))
    Wu = r.standard_normal((h, f))
    bu = r.standard_normal(f)
    cst = 0.8
    W1 = np.concatenate([np.zeros((h, f)), Wu], axis=1)
    b1 = np.concatenate([np.full(f, cst), bu])
    W2 = r.standard_normal((f, h))
    out = oracle.swiglu_forward(X, W1, b1, W2, None)
    Y = cst * expit(cst) * (X @ Wu + bu)
    np.testing.assert_allclose(out["Y"], Y, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out["Z"], Y @ W2, rtol=1e-12, atol=1e-12)


def _swiglu_loss(X, W1, b1, W2, b2, dZ):
    return float(np.sum(dZ * oracle.swiglu_forward(X, W1, b1, W2, b2)["Z"]))


def test_swiglu_backward_matches_finite_differences():
    T, h, f = 3, 4, 5
    r = rng(23)
    P = {"X": r.standard_normal((T, h)), "W1": 0.6 * r.standard_normal((h, 2 * f)),
         "b1": 0.3 * r.standard_normal(2 * f), "W2": 0.5 * r.standard_normal((f, h)),
         "b2": 0.3 * r.standard_normal(h)}
    dZ = r.standard_normal((T, h))
    g = oracle.swiglu_backward(P["X"], P["W1"], P["b1"], P["W2"], dZ)
    grads = {"X": g["dX"], "W1": g["dW1"], "b1": g["db1"], "W2": g["dW2"], "b2": g["db2"]}
    e = 1e-5
    for name, val in P.items():
        fd = np.zeros_like(val)
        for idx in np.ndindex(val.shape):
            plus = {k: v.copy() for k, v in P.items()}
            minus = {k: v.copy() for k, v in P.items()}
            plus[name][idx] += e
            minus[name][idx] -= e
            fd[idx] = (_swiglu_loss(**plus, dZ=dZ) - _swiglu_loss(**minus, dZ=dZ)) / (2 * e)
        scale = max(1.0, np.abs(fd).max())
        assert np.abs(fd - grads[name]).max() < 1e-7 * scale, name


def test_swiglu_backward_cols_match_full_backward():
    T, h, f = 5, 6, 8
    r = rng(24)
    X, W1, W2 = r.standard_normal((T, h)), r.standard_normal((h, 2 * f)), r.standard_normal((f, h))
    b1, dZ = r.standard_normal(2 * f), r.standard_normal((T, h))
    full = oracle.swiglu_backward(X, W1, b1, W2, dZ)
    cols = [0, 5, 7]
    part = oracle.swiglu_backward_cols(X, W1, b1, W2, dZ, cols)
    up = [f + c for c in cols]
    np.testing.assert_allclose(part["dW1_gate"], full["dW1"][:, cols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(part["dW1_up"], full["dW1"][:, up], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(part["db1_gate"], full["db1"][cols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(part["db1_up"], full["db1"][up], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(part["dW2"], full["dW2"][cols, :], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("t", [1, 2, 3, 6])
def test_swiglu_sharded_equals_unsharded(t):
    T, h, f = 4, 5, 6
    r = rng(25)
    X, W1, W2 = r.standard_normal((T, h)), r.standard_normal((h, 2 * f)), r.standard_normal((f, h))
    b1, b2, dZ = r.standard_normal(2 * f), r.standard_normal(h), r.standard_normal((T, h))
    ref_f = oracle.swiglu_forward(X, W1, b1, W2, b2)
    ref_b = oracle.swiglu_backward(X, W1, b1, W2, dZ)
    sh = oracle.swiglu_sharded(X, W1, b1, W2, b2, dZ, t)
    np.testing.assert_allclose(sh["Z"], ref_f["Z"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sh["dX"], ref_b["dX"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sh["dW1"], ref_b["dW1"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sh["dW2"], ref_b["dW2"], rtol=1e-12, atol=1e-12)
