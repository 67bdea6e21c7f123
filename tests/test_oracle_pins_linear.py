"""Pins for the linear-layer part of the CPU oracle: the ColumnParallelLinear
and RowParallelLinear primitives of the 70B page ("The Mechanics of Tensor
Parallelism (TP) in Megatron-LM") and the fused QKV head layout of its
"The Multi-Head Attention Block" section.

Checked against numpy's matmul (a library routine), central differences of
the oracle's own forward, the partition algebra (sharded == unsharded in both
modes, the row-parallel bias once) and the page's own head count per GPU
(tests/golden/gqa_heads_per_shard.txt).
"""

import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def rng(seed):
    return np.random.default_rng(seed)


def test_linear_forward_matches_numpy_matmul():
    r = rng(31)
    X, W, b = r.standard_normal((5, 7)), r.standard_normal((7, 3)), r.standard_normal(3)
    np.testing.assert_allclose(oracle.linear_forward(X, W, b), X @ W + b, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.linear_forward(X, W), X @ W, rtol=1e-13, atol=1e-13)


def test_linear_forward_with_permutation_weights():
    # column j of W picks input p[j] scaled by c[j]: Y[:, j] = c[j] X[:, p[j]] + b[j]
    r = rng(32)
    X = r.standard_normal((4, 6))
    p, c, b = r.integers(0, 6, size=9), r.uniform(-2, 2, size=9), r.standard_normal(9)
    W = np.zeros((6, 9))
    W[p, np.arange(9)] = c
    np.testing.assert_allclose(oracle.linear_forward(X, W, b), c * X[:, p] + b, atol=1e-14)


def test_linear_backward_matches_finite_differences():
    r = rng(33)
    X, W, b, dY = r.standard_normal((3, 4)), r.standard_normal((4, 5)), r.standard_normal(5), r.standard_normal((3, 5))
    g = oracle.linear_backward(X, W, dY)

    def loss(X_, W_, b_):
        return float(np.sum(dY * oracle.linear_forward(X_, W_, b_)))

    e = 1e-6
    for name, val, grad in (("X", X, g["dX"]), ("W", W, g["dW"]), ("b", b, g["db"])):
        fd = np.zeros_like(val)
        for idx in np.ndindex(val.shape):
            P = {"X_": X.copy(), "W_": W.copy(), "b_": b.copy()}
            M = {"X_": X.copy(), "W_": W.copy(), "b_": b.copy()}
            P[name + "_"][idx] += e
            M[name + "_"][idx] -= e
            fd[idx] = (loss(**P) - loss(**M)) / (2 * e)
        assert np.abs(fd - grad).max() < 1e-7 * max(1.0, np.abs(fd).max()), name


@pytest.mark.parametrize("mode", ["column", "row"])
@pytest.mark.parametrize("t", [1, 2, 3, 6])
def test_linear_sharded_equals_unsharded(mode, t):
    r = rng(34)
    X, W, b, dY = r.standard_normal((4, 12)), r.standard_normal((12, 6)), r.standard_normal(6), r.standard_normal((4, 6))
    sh = oracle.linear_sharded(X, W, b, dY, t, mode)
    ref = oracle.linear_backward(X, W, dY)
    np.testing.assert_allclose(sh["Y"], oracle.linear_forward(X, W, b), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sh["dX"], ref["dX"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sh["dW"], ref["dW"], rtol=1e-12, atol=1e-12)


def test_row_parallel_linear_bias_enters_once():
    r = rng(35)
    b = r.standard_normal(4)
    for t in (1, 2, 4):
        sh = oracle.linear_sharded(r.standard_normal((3, 8)), np.zeros((8, 4)), b, np.zeros((3, 4)), t, "row")
        np.testing.assert_allclose(sh["Y"], np.broadcast_to(b, (3, 4)), atol=0)


def _golden_heads():
    rows = []
    for line in open(os.path.join(HERE, "golden", "gqa_heads_per_shard.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(tuple(int(x) for x in line.split()))
    return rows


def _owners(cols, width, t):
    return np.unique(cols // (width // t))


@pytest.mark.parametrize("n_q,n_kv,t,qps,kvps", _golden_heads())
def test_qkv_layout_gives_each_shard_whole_heads_page_example(n_q, n_kv, t, qps, kvps):
    d = 4  # the head width does not change which heads a shard holds
    width = (n_q + 2 * n_kv) * d
    q, k, v = (oracle.qkv_columns(kind, n_q, n_kv, d) for kind in ("q", "k", "v"))
    # a bijection onto [0, width)
    allc = np.concatenate([q.ravel(), k.ravel(), v.ravel()])
    assert np.array_equal(np.sort(allc), np.arange(width))
    for i in range(t):
        mine_q = [hh for hh in range(n_q) if list(_owners(q[hh], width, t)) == [i]]
        mine_k = [hh for hh in range(n_kv) if list(_owners(k[hh], width, t)) == [i]]
        mine_v = [hh for hh in range(n_kv) if list(_owners(v[hh], width, t)) == [i]]
        assert len(mine_q) == qps and len(mine_k) == kvps and mine_k == mine_v
        # a shard's query heads are those that share its key/value heads
        assert all(hh // (n_q // n_kv) in mine_k for hh in mine_q)


@pytest.mark.parametrize("n_q,n_kv,t", [(8, 2, 2), (12, 4, 4), (6, 6, 3), (4, 1, 1)])
def test_qkv_projection_splits_into_per_head_products(n_q, n_kv, t):
    # pack separate W_Q, W_K, W_V by the layout, project once, and read the
    # heads back: each equals X W for its own weight (numpy matmul)
    d, h, T = 3, 5, 4
    r = rng(36)
    X = r.standard_normal((T, h))
    Wq, Wk, Wv = r.standard_normal((h, n_q * d)), r.standard_normal((h, n_kv * d)), r.standard_normal((h, n_kv * d))
    q, k, v = (oracle.qkv_columns(kind, n_q, n_kv, d) for kind in ("q", "k", "v"))
    W = np.zeros((h, (n_q + 2 * n_kv) * d))
    W[:, q.ravel()] = Wq
    W[:, k.ravel()] = Wk
    W[:, v.ravel()] = Wv
    QKV = oracle.linear_forward(X, W)
    np.testing.assert_allclose(QKV[:, q.ravel()], X @ Wq, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(QKV[:, k.ravel()], X @ Wk, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(QKV[:, v.ravel()], X @ Wv, rtol=1e-12, atol=1e-12)
    # the column-parallel split: shard i's contiguous block is its heads' projection
    width = W.shape[1]
    sh = oracle.linear_sharded(X, W, None, np.zeros((T, width)), t, "column")
    np.testing.assert_allclose(sh["Y"], QKV, rtol=1e-12, atol=1e-12)
