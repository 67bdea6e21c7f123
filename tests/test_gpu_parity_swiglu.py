"""GPU parity of the SwiGLU block (tp_swiglu_forward / tp_swiglu_backward)
against the fp64 CPU oracle, every output element, through the C ABI.

Cases span several gated tiles (128 output columns each on the bf16 path, 64
on the tf32 path), ragged T and h, an f whose last gated tile is partly
outside [0, f) (its gate half then overlaps the up columns and its up half
runs past 2f), one token, and non-zero biases on both halves.
"""

import numpy as np
import pytest
import torch

import oracle
import vocab_ce_gb300 as tp
from vocab_ce_gb300 import workloads as wl
from _parity import assert_rel, gpu_or_skip

pytestmark = pytest.mark.gpu


def _biases(w, seed):
    g = torch.Generator().manual_seed(2000 + seed)
    return (0.1 * torch.randn(2 * w.f, generator=g)).float(), (0.1 * torch.randn(w.h, generator=g)).float()


def run_swiglu(w, dev, seed=0, nonzero_bias=True):
    si = wl.swiglu_inputs(w, seed=seed)
    if nonzero_bias:
        si["b1"], si["b2"] = _biases(w, seed)
    g = {k: v.to(dev) for k, v in si.items()}
    fwd = tp.tp_swiglu_forward(g["X"], g["W1"], g["W2"], w.t, g["b1"], g["b2"])
    bwd = tp.tp_swiglu_backward(g["dZ"], g["X"], g["W1"], g["W2"], fwd["GU"], fwd["Y"], w.t)
    assert tp.device_status() == 0
    return si, fwd, bwd


SWIGLU_CASES = {
    # name: (T, h, f, t, dtype)
    "tiny_shape_f32": (32, 64, 256, 2, "f32"),
    "tiny_shape_bf16": (32, 64, 256, 2, "bf16"),
    "ragged": (333, 200, 384, 2, "bf16"),
    "multi_tile": (640, 512, 1024, 4, "bf16"),
    "ragged_gated_tile": (300, 136, 320, 5, "bf16"),   # f = 320: the third 128-column tile is half outside
    "one_token": (1, 64, 128, 2, "bf16"),
    "wide": (1000, 1536, 3072, 8, "bf16"),
    "ragged_f32": (333, 200, 384, 2, "f32"),
    "multi_tile_f32": (300, 256, 512, 4, "f32"),
    "odd_shards_f32": (70, 64, 192, 3, "f32"),
}


@pytest.mark.parametrize("case", list(SWIGLU_CASES))
def test_swiglu_matches_oracle(case):
    dev = gpu_or_skip()
    T, h, f, t, dtype = SWIGLU_CASES[case]
    w = wl.custom(case, T=T, h=h, f=f, v_valid=0, v_pad=0, t=t, dtype=dtype, act="swiglu")
    si, fwd, bwd = run_swiglu(w, dev)
    of = oracle.swiglu_forward(si["X"], si["W1"], si["b1"], si["W2"], si["b2"])
    ob = oracle.swiglu_backward(si["X"], si["W1"], si["b1"], si["W2"], si["dZ"])
    assert_rel("G", fwd["GU"][:, :f], of["GU"][:, :f])
    assert_rel("Up", fwd["GU"][:, f:], of["GU"][:, f:])
    for k in ("Y", "Z"):
        assert_rel(k, fwd[k], of[k])
    assert_rel("dW1 gate", bwd["dW1"][:, :f], ob["dW1"][:, :f])
    assert_rel("dW1 up", bwd["dW1"][:, f:], ob["dW1"][:, f:])
    assert_rel("db1 gate", bwd["db1"][:f], ob["db1"][:f])
    assert_rel("db1 up", bwd["db1"][f:], ob["db1"][f:])
    for k in ("dX", "dW2", "db2"):
        assert_rel(k, bwd[k], ob[k])


def test_swish_and_derivative_evaluation_error_fp32():
    # Swish and Swish' on the device checked at their own accuracy through the
    # fp32 API: W1 = [I | 0], b1 = [0 | 1] gives G = tf32(X), Up = 1 and
    # Y = Swish(G); W2 = I and dZ = 1 on one token give dY = 1, so
    # db1[:f] = Swish'(G) and db1[f:] = Swish(G), up to the device evaluation.
    dev = gpu_or_skip()
    h = f = 256
    X = torch.linspace(-12.0, 12.0, h, dtype=torch.float32).reshape(1, h).to(dev)
    I = torch.eye(h, dtype=torch.float32, device=dev)
    W1 = torch.cat([I, torch.zeros_like(I)], dim=1).contiguous()
    b1 = torch.cat([torch.zeros(f), torch.ones(f)]).float().to(dev)
    fwd = tp.tp_swiglu_forward(X, W1, I, 2, b1)
    bwd = tp.tp_swiglu_backward(torch.ones(1, h, device=dev), X, W1, I, fwd["GU"], fwd["Y"], 2)
    assert tp.device_status() == 0
    G = fwd["GU"].double().cpu().numpy()[0, :f]
    Y = fwd["Y"].double().cpu().numpy()[0]
    db1 = bwd["db1"].double().cpu().numpy()
    sw = np.array([oracle.swish(g) for g in G])
    dsw = np.array([oracle.swish_grad(g) for g in G])
    assert np.abs(Y - sw).max() <= 2e-6 * max(1.0, np.abs(G).max())
    assert np.abs(db1[f:] - sw).max() <= 2e-6 * max(1.0, np.abs(G).max())
    assert np.abs(db1[:f] - dsw).max() <= 2e-6


def test_swish_saturated_gates_fp32():
    # |G| up to 120: exp overflows inside the sigmoid, which must still give the
    # limits Swish -> 0 (G << 0), G (G >> 0) and Swish' -> 0, 1, with no NaN
    dev = gpu_or_skip()
    h = f = 256
    X = torch.linspace(-120.0, 120.0, h, dtype=torch.float32).reshape(1, h).to(dev)
    I = torch.eye(h, dtype=torch.float32, device=dev)
    W1 = torch.cat([I, torch.zeros_like(I)], dim=1).contiguous()
    b1 = torch.cat([torch.zeros(f), torch.ones(f)]).float().to(dev)
    fwd = tp.tp_swiglu_forward(X, W1, I, 2, b1)
    bwd = tp.tp_swiglu_backward(torch.ones(1, h, device=dev), X, W1, I, fwd["GU"], fwd["Y"], 2)
    assert tp.device_status() == 0
    G = fwd["GU"].double().cpu().numpy()[0, :f]
    Y = fwd["Y"].double().cpu().numpy()[0]
    db1 = bwd["db1"].double().cpu().numpy()
    assert np.isfinite(Y).all() and np.isfinite(db1).all()
    sw = np.array([oracle.swish(g) for g in G])
    dsw = np.array([oracle.swish_grad(g) for g in G])
    assert np.abs(Y - sw).max() <= 2e-6 * np.abs(G).max()
    assert np.abs(db1[f:] - sw).max() <= 2e-6 * np.abs(G).max()
    assert np.abs(db1[:f] - dsw).max() <= 2e-6


def test_swiglu_shard_count_does_not_change_results():
    dev = gpu_or_skip()
    base = None
    for t in (1, 2, 4, 8):
        w = wl.custom(f"t{t}", T=512, h=256, f=1024, v_valid=0, v_pad=0, t=t, act="swiglu")
        si, fwd, bwd = run_swiglu(w, dev)
        cur = {**{k: fwd[k].cpu() for k in ("Z", "GU", "Y")}, **{k: v.cpu() for k, v in bwd.items()}}
        if base is None:
            base = cur
            of = oracle.swiglu_forward(si["X"], si["W1"], si["b1"], si["W2"], si["b2"])
            assert_rel("Z", fwd["Z"], of["Z"])
        else:
            for k in base:
                assert torch.equal(base[k], cur[k]), f"t={t}: {k} differs from t=1"


def test_swiglu_empty_batch():
    dev = gpu_or_skip()
    h, f = 64, 128
    X = torch.empty((0, h), dtype=torch.bfloat16, device=dev)
    W1 = torch.randn(h, 2 * f, device=dev).bfloat16()
    W2 = torch.randn(f, h, device=dev).bfloat16()
    fwd = tp.tp_swiglu_forward(X, W1, W2, 2)
    assert fwd["Z"].shape == (0, h)
    bwd = tp.tp_swiglu_backward(X, X, W1, W2, fwd["GU"], fwd["Y"], 2)
    assert tp.device_status() == 0
    for k in ("dW1", "dW2", "db1", "db2"):
        assert torch.count_nonzero(bwd[k]).item() == 0, k
