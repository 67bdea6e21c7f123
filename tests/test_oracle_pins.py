"""Pins for the CPU oracle, checked against what the pages and the mathematics
fix rather than against the oracle itself: closed forms, special cases that
reduce to library routines (scipy's normal CDF and logsumexp), finite
differences of the oracle's own forward, and the partition algebra of the
Megatron pages (sharded == unsharded for every t).

Each pin is chosen so that a plausible slip in ``oracle/oracle.c`` fails it:
a transposed or wrongly indexed operand (permutation weights, h != f), a
dropped or misplaced bias (non-zero biases, bias added once after the shard
sum), a wrong sign or derivative (finite differences), a missing max
subtraction (a logit of 800), padded ids leaking into the loss (padded rows of
E set large, loss = ln v_valid), a wrong shard combine (t up to 16 with
all-padding shards).
"""

import math

import numpy as np
import pytest
from scipy.special import logsumexp
from scipy.stats import norm

import oracle


def rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# GeLU
# --------------------------------------------------------------------------

def test_gelu_special_values():
    # GeLU(0) = 0, GeLU'(0) = 1/2 (closed form of x * Phi(x))
    assert oracle.gelu(0.0) == 0.0
    assert abs(oracle.gelu_grad(0.0) - 0.5) < 1e-15


@pytest.mark.parametrize("x", [-6.0, -2.5, -1.0, -0.3, 0.7, 1.0, 2.0, 4.5])
def test_gelu_is_x_times_normal_cdf(x):
    # the exact (erf) GeLU equals x * Phi(x) with scipy's normal CDF
    assert abs(oracle.gelu(x) - x * norm.cdf(x)) < 1e-14 * max(1.0, abs(x))


@pytest.mark.parametrize("x", [-3.0, -1.0, -0.25, 0.5, 1.5, 3.0])
def test_gelu_odd_part_identity(x):
    # Phi(-x) = 1 - Phi(x)  =>  GeLU(x) - GeLU(-x) = x
    assert abs(oracle.gelu(x) - oracle.gelu(-x) - x) < 1e-14 * max(1.0, abs(x))


@pytest.mark.parametrize("x", [-2.0, -0.5, 0.1, 1.3, 2.7])
def test_gelu_grad_matches_central_difference(x):
    e = 1e-5
    fd = (oracle.gelu(x + e) - oracle.gelu(x - e)) / (2 * e)
    assert abs(fd - oracle.gelu_grad(x)) < 1e-9
    # and the closed form Phi(x) + x phi(x) via scipy
    assert abs(oracle.gelu_grad(x) - (norm.cdf(x) + x * norm.pdf(x))) < 1e-14


# --------------------------------------------------------------------------
# MLP forward: permutation weights reduce the products to indexing
# --------------------------------------------------------------------------

def test_mlp_forward_with_permutation_weights():
    T, h, f = 4, 5, 10
    r = rng(1)
    X = r.standard_normal((T, h))
    pi = r.integers(0, h, size=f)             # column j of A picks input pi[j]
    d = r.uniform(0.5, 2.0, size=f)
    A = np.zeros((h, f))
    A[pi, np.arange(f)] = d
    bA = r.standard_normal(f)
    sigma = r.permutation(f)[:h]              # output n reads hidden unit sigma[n]
    c = r.uniform(-2.0, 2.0, size=h)
    B = np.zeros((f, h))
    B[sigma, np.arange(h)] = c
    bB = r.standard_normal(h)

    out = oracle.mlp_forward(X, A, bA, B, bB)
    U_exp = d[None, :] * X[:, pi] + bA[None, :]
    Y_exp = U_exp * norm.cdf(U_exp)
    Z_exp = c[None, :] * Y_exp[:, sigma] + bB[None, :]
    np.testing.assert_allclose(out["U"], U_exp, rtol=0, atol=1e-14)
    np.testing.assert_allclose(out["Y"], Y_exp, rtol=0, atol=1e-13)
    np.testing.assert_allclose(out["Z"], Z_exp, rtol=0, atol=1e-13)


def test_mlp_identity_weights_give_gelu_of_input():
    # A = I, bA = 0 gives Y = GeLU(X); B = I gives Z = Y
    T, h = 3, 6
    X = rng(2).standard_normal((T, h))
    I = np.eye(h)
    out = oracle.mlp_forward(X, I, None, I, None)
    np.testing.assert_allclose(out["Y"], X * norm.cdf(X), atol=1e-14)
    np.testing.assert_allclose(out["Z"], out["Y"], atol=0)


def test_mlp_zero_input_exposes_biases():
    # X = 0: U = bA, Z = GeLU(bA) B + bB
    T, h, f = 2, 3, 4
    r = rng(3)
    bA = r.standard_normal(f)
    bB = r.standard_normal(h)
    B = np.zeros((f, h))
    B[1, 2] = 3.0
    out = oracle.mlp_forward(np.zeros((T, h)), r.standard_normal((h, f)), bA, B, bB)
    np.testing.assert_allclose(out["U"], np.broadcast_to(bA, (T, f)), atol=0)
    z = np.broadcast_to(bB, (T, h)).copy()
    z[:, 2] += 3.0 * bA[1] * norm.cdf(bA[1])
    np.testing.assert_allclose(out["Z"], z, atol=1e-14)


# --------------------------------------------------------------------------
# MLP backward: central differences of the oracle's own forward
# --------------------------------------------------------------------------

def _mlp_loss(X, A, bA, B, bB, dZ):
    return float(np.sum(dZ * oracle.mlp_forward(X, A, bA, B, bB)["Z"]))


def test_mlp_backward_matches_finite_differences():
    T, h, f = 3, 4, 6
    r = rng(4)
    P = {"X": r.standard_normal((T, h)), "A": 0.5 * r.standard_normal((h, f)),
         "bA": 0.3 * r.standard_normal(f), "B": 0.5 * r.standard_normal((f, h)),
         "bB": 0.3 * r.standard_normal(h)}
    dZ = r.standard_normal((T, h))
    g = oracle.mlp_backward(P["X"], P["A"], P["bA"], P["B"], dZ)
    grads = {"X": g["dX"], "A": g["dA"], "bA": g["dbA"], "B": g["dB"], "bB": g["dbB"]}
    e = 1e-5
    for name, val in P.items():
        fd = np.zeros_like(val)
        for idx in np.ndindex(val.shape):
            plus = {k: v.copy() for k, v in P.items()}
            minus = {k: v.copy() for k, v in P.items()}
            plus[name][idx] += e
            minus[name][idx] -= e
            fd[idx] = (_mlp_loss(**plus, dZ=dZ) - _mlp_loss(**minus, dZ=dZ)) / (2 * e)
        scale = max(1.0, np.abs(fd).max())
        assert np.abs(fd - grads[name]).max() < 1e-7 * scale, name


def test_bias_grad_is_token_sum():
    # dbB of the block equals the column sums of dZ: with B = 0 the loss
    # sum(dZ * Z) is sum(dZ * bB), whose gradient in bB is sum_t dZ
    T, h, f = 6, 5, 4
    r = rng(16)
    dZ = r.standard_normal((T, h))
    g = oracle.mlp_backward(r.standard_normal((T, h)), r.standard_normal((h, f)), None,
                            np.zeros((f, h)), dZ)
    np.testing.assert_allclose(oracle.bias_grad(dZ), g["dbB"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(oracle.bias_grad(np.ones((T, h))), np.full(h, float(T)), atol=0)


def test_mlp_backward_cols_match_full_backward():
    T, h, f = 5, 6, 10
    r = rng(5)
    X, A, B = r.standard_normal((T, h)), r.standard_normal((h, f)), r.standard_normal((f, h))
    bA, dZ = r.standard_normal(f), r.standard_normal((T, h))
    full = oracle.mlp_backward(X, A, bA, B, dZ)
    cols = [0, 3, 9]
    part = oracle.mlp_backward_cols(X, A, bA, B, dZ, cols)
    np.testing.assert_allclose(part["dA"], full["dA"][:, cols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(part["dbA"], full["dbA"][cols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(part["dB"], full["dB"][cols, :], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# The partition algebra: column-parallel A, row-parallel B, g and f*
# --------------------------------------------------------------------------

@pytest.mark.parametrize("t", [1, 2, 3, 4, 6, 12])
def test_mlp_sharded_equals_unsharded(t):
    T, h, f = 4, 5, 12
    r = rng(6)
    X, A, B = r.standard_normal((T, h)), r.standard_normal((h, f)), r.standard_normal((f, h))
    bA, bB, dZ = r.standard_normal(f), r.standard_normal(h), r.standard_normal((T, h))
    ref_f = oracle.mlp_forward(X, A, bA, B, bB)
    ref_b = oracle.mlp_backward(X, A, bA, B, dZ)
    sh = oracle.mlp_sharded(X, A, bA, B, bB, dZ, t)
    np.testing.assert_allclose(sh["Z"], ref_f["Z"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sh["dX"], ref_b["dX"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sh["dA"], ref_b["dA"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sh["dB"], ref_b["dB"], rtol=1e-12, atol=1e-12)


def test_row_parallel_bias_enters_once():
    # with B = 0 every shard's partial is zero, so Z = bB for every t
    T, h, f = 2, 3, 8
    r = rng(7)
    bB = r.standard_normal(h)
    for t in (1, 2, 4, 8):
        sh = oracle.mlp_sharded(r.standard_normal((T, h)), r.standard_normal((h, f)),
                                r.standard_normal(f), np.zeros((f, h)), bB,
                                np.zeros((T, h)), t)
        np.testing.assert_allclose(sh["Z"], np.broadcast_to(bB, (T, h)), atol=0)


# --------------------------------------------------------------------------
# Cross-entropy
# --------------------------------------------------------------------------

def test_ce_zero_embedding_gives_log_vocab_and_masks_padding():
    # E = 0 on the real ids makes every logit 0: loss = ln(v_valid). The padded
    # rows are set large; they must not enter (ln 128,256, not ln 129,024).
    T, h, v_valid, v_pad = 3, 4, 128256, 129024
    r = rng(8)
    H = r.standard_normal((T, h))
    E = np.zeros((v_pad, h))
    E[v_valid:] = 30.0
    y = np.array([0, 77777, v_valid - 1], dtype=np.int32)
    gs = 0.5
    out = oracle.ce(H, E, y, v_valid, grad_scale=gs)
    assert math.log(v_pad) - math.log(v_valid) > 5e-3  # the two readings are distinguishable
    np.testing.assert_allclose(out["loss"], math.log(v_valid), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["lse"], math.log(v_valid), rtol=0, atol=1e-12)
    # dH = sum_j dl_j E_j = 0 on the real ids
    np.testing.assert_allclose(out["dH"], 0.0, atol=0)
    # dE_v = gs * sum_t (1/v_valid - [v == y_t]) H_t on real ids, 0 on padded ids
    dE = out["dE"]
    colsum = H.sum(axis=0)
    expect_rest = gs * colsum / v_valid
    rest = np.ones(v_pad, dtype=bool)
    rest[y] = False
    rest[v_valid:] = False
    np.testing.assert_allclose(dE[rest], np.broadcast_to(expect_rest, dE[rest].shape), rtol=1e-12, atol=1e-18)
    for t_ in range(T):
        np.testing.assert_allclose(dE[y[t_]], expect_rest - gs * H[t_], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dE[v_valid:], 0.0, atol=0)


@pytest.mark.parametrize("c", [0.0, 5.0, -3.0, 800.0])
def test_ce_single_token_closed_form(c):
    # T = 1, E_target = c H / |H|^2, other rows 0: l_target = c, other logits 0,
    # loss = ln(v_valid - 1 + e^c) - c = log1p((v_valid - 1) e^-c). c = 800
    # overflows exp(l) without the max subtraction.
    h, v_valid, v_pad = 6, 1000, 1024
    r = rng(9)
    Hrow = r.standard_normal(h)
    E = np.zeros((v_pad, h))
    y = 417
    E[y] = c * Hrow / float(Hrow @ Hrow)
    out = oracle.ce(Hrow[None, :], E, np.array([y], dtype=np.int32), v_valid, grads=False)
    expect = math.log1p((v_valid - 1) * math.exp(-c)) if c > 0 else math.log(v_valid - 1 + math.exp(c)) - c
    assert abs(out["loss"][0] - expect) < 1e-12 * max(1.0, abs(expect))


def test_ce_matches_library_logsumexp():
    T, h, v_valid, v_pad = 7, 5, 50, 64
    r = rng(10)
    H, E = r.standard_normal((T, h)), r.standard_normal((v_pad, h))
    y = r.integers(0, v_valid, size=T).astype(np.int32)
    out = oracle.ce(H, E, y, v_valid, grads=False)
    logits = np.matmul(H, E[:v_valid].T)
    lse = logsumexp(logits, axis=1)
    np.testing.assert_allclose(out["lse"], lse, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out["loss"], lse - logits[np.arange(T), y], rtol=1e-12, atol=1e-12)


def test_ce_gradients_match_finite_differences():
    T, h, v_valid, v_pad = 3, 4, 13, 16
    r = rng(11)
    H, E = r.standard_normal((T, h)), r.standard_normal((v_pad, h))
    y = np.array([0, 12, 5], dtype=np.int32)
    gs = 0.7
    out = oracle.ce(H, E, y, v_valid, grad_scale=gs)

    def L(Hm, Em):
        return gs * float(oracle.ce(Hm, Em, y, v_valid, grads=False)["loss"].sum())

    e = 1e-5
    for name, val, grad in (("H", H, out["dH"]), ("E", E, out["dE"])):
        fd = np.zeros_like(val)
        for idx in np.ndindex(val.shape):
            p, m = val.copy(), val.copy()
            p[idx] += e
            m[idx] -= e
            fd[idx] = (L(p, E) - L(m, E)) / (2 * e) if name == "H" else (L(H, p) - L(H, m)) / (2 * e)
        assert np.abs(fd - grad).max() < 1e-8 * max(1.0, np.abs(fd).max()), name
    # padded rows get no gradient at all
    np.testing.assert_allclose(out["dE"][v_valid:], 0.0, atol=0)


def test_ce_gradient_rows_sum_to_zero():
    # sum_j (softmax_j - onehot_j) = 0 for every token, hence sum_v dE_v = 0
    T, h, v_valid, v_pad = 9, 7, 90, 96
    r = rng(12)
    H, E = r.standard_normal((T, h)), 0.3 * r.standard_normal((v_pad, h))
    y = r.integers(0, v_valid, size=T).astype(np.int32)
    out = oracle.ce(H, E, y, v_valid, grad_scale=1.0)
    np.testing.assert_allclose(out["dE"].sum(axis=0), 0.0, atol=1e-12)


@pytest.mark.parametrize("t", [1, 2, 4, 8, 16])
def test_ce_shard_combine_equals_unsharded(t):
    # v_pad = 128, v_valid = 100: at t = 16 the shards 13..15 hold only padding
    T, h, v_valid, v_pad = 11, 6, 100, 128
    r = rng(13)
    H, E = r.standard_normal((T, h)), r.standard_normal((v_pad, h))
    y = r.integers(0, v_valid, size=T).astype(np.int32)
    y[0], y[1] = 0, v_valid - 1
    ref = oracle.ce(H, E, y, v_valid, grads=False)
    sh = oracle.ce_sharded(H, E, y, v_valid, t)
    np.testing.assert_allclose(sh["loss"], ref["loss"], rtol=0, atol=1e-12)
    vs = v_pad // t
    for i in range(t):
        if i * vs >= v_valid:
            assert np.all(np.isneginf(sh["m"][i])) and np.all(sh["s"][i] == 0.0)
    # the target logit comes from exactly one shard
    logits = H @ E.T
    np.testing.assert_allclose(sh["tau"], logits[np.arange(T), y], rtol=1e-13, atol=1e-13)


def test_ce_out_of_range_target_is_nan():
    H, E = rng(14).standard_normal((2, 3)), rng(15).standard_normal((8, 3))
    out = oracle.ce(H, E, np.array([1, 6], dtype=np.int32), 6, grads=False)
    assert np.isfinite(out["loss"][0]) and np.isnan(out["loss"][1])


def test_oracle_reports_threads():
    assert oracle.num_threads() >= 1


# --------------------------------------------------------------------------
# Sequence parallelism: all-gather entry, reduce-scatter exit
# --------------------------------------------------------------------------

@pytest.mark.parametrize("t", [1, 2, 3, 6])
def test_seq_parallel_equals_unsharded_rows(t):
    # the reduce-scatter exit hands rank r exactly rows r of the all-reduced Z
    # ("All-Reduce = Reduce-Scatter + All-Gather"), and the backward's dX chunks
    # are the rows of the unsharded dX; the weight gradients are unchanged
    T, h, f = 12, 5, 12
    r = rng(41)
    X, A, B = r.standard_normal((T, h)), r.standard_normal((h, f)), r.standard_normal((f, h))
    bA, bB, dZ = r.standard_normal(f), r.standard_normal(h), r.standard_normal((T, h))
    rows = T // t
    sp = oracle.mlp_seq_parallel([X[i * rows:(i + 1) * rows] for i in range(t)], A, bA, B, bB,
                                 [dZ[i * rows:(i + 1) * rows] for i in range(t)])
    ref_f = oracle.mlp_forward(X, A, bA, B, bB)
    ref_b = oracle.mlp_backward(X, A, bA, B, dZ)
    np.testing.assert_allclose(np.concatenate(sp["Z"]), ref_f["Z"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(np.concatenate(sp["dX"]), ref_b["dX"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sp["dA"], ref_b["dA"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sp["dB"], ref_b["dB"], rtol=1e-12, atol=1e-12)


def test_seq_parallel_chunk_order_matters():
    # permuting the X chunks permutes the Z chunks the same way (the exit is a
    # scatter by sequence position, not a sum over chunks)
    T, h, f, t = 8, 4, 8, 4
    r = rng(42)
    X, A, B = r.standard_normal((T, h)), r.standard_normal((h, f)), r.standard_normal((f, h))
    dZ = r.standard_normal((T, h))
    chunks = [X[i * 2:(i + 1) * 2] for i in range(t)]
    dzc = [dZ[i * 2:(i + 1) * 2] for i in range(t)]
    perm = [2, 0, 3, 1]
    a = oracle.mlp_seq_parallel(chunks, A, None, B, None, dzc)
    b = oracle.mlp_seq_parallel([chunks[p] for p in perm], A, None, B, None, [dzc[p] for p in perm])
    for k, p in enumerate(perm):
        np.testing.assert_allclose(b["Z"][k], a["Z"][p], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(b["dX"][k], a["dX"][p], rtol=1e-12, atol=1e-12)
