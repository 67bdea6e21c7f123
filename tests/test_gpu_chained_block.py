"""The block chained into the vocabulary-parallel loss, as a training step of
the last layer and the head uses it: Z = MLP(X) is the CE input H, and the
CE's dH is the MLP's upstream gradient dZ. Compared with the same chain in the
fp64 oracle (which does not round Z or dH to bf16 between the stages; the
tolerance absorbs that). Also the forward-only loss on the chained input (the
evaluation use).
"""

import numpy as np
import pytest
import torch

import oracle
import vocab_ce_gb300 as tp
from vocab_ce_gb300 import workloads as wl
from _parity import assert_loss, assert_rel, gpu_or_skip

pytestmark = pytest.mark.gpu


def chained(w, dev, seed=0, gs=None):
    mi = wl.mlp_inputs(w, seed=seed, device=dev)
    ci = wl.ce_inputs(w, seed=seed, device=dev)
    gs = 1.0 / w.T if gs is None else gs
    fwd = tp.tp_mlp_forward(mi["X"], mi["A"], mi["B"], w.t, mi["bA"], mi["bB"])
    ce = tp.vocab_parallel_ce(fwd["Z"], ci["E"], ci["targets"], w.v_valid, w.t, grad_scale=gs)
    bwd = tp.tp_mlp_backward(ce["dH"], mi["X"], mi["A"], mi["B"], fwd["U"], fwd["Y"], w.t)
    ev = tp.vocab_parallel_ce(fwd["Z"], ci["E"], ci["targets"], w.v_valid, w.t, grads=False)
    assert tp.device_status() == 0
    return mi, ci, fwd, ce, bwd, ev, gs


def test_chained_block_and_loss_small():
    dev = gpu_or_skip()
    w = wl.custom("chain", T=300, h=256, f=1024, v_valid=1900, v_pad=2048, t=4)
    mi, ci, fwd, ce, bwd, ev, gs = chained(w, dev)
    h = {k: v.cpu() for k, v in {**mi, **ci}.items()}
    of = oracle.mlp_forward(h["X"], h["A"], h["bA"], h["B"], h["bB"])
    oc = oracle.ce(of["Z"], h["E"], h["targets"].numpy(), w.v_valid, grad_scale=gs)
    ob = oracle.mlp_backward(h["X"], h["A"], h["bA"], h["B"], oc["dH"])
    assert_loss("loss", ce["loss"], oc["loss"])
    assert_loss("eval loss", ev["loss"], oc["loss"])
    assert torch.equal(ev["loss"], ce["loss"]), "the forward-only loss equals the training loss bit for bit"
    assert_rel("dH = dZ", ce["dH"], oc["dH"])
    assert_rel("dE", ce["dE"], oc["dE"])
    for k in ("dX", "dA", "dB", "dbA", "dbB"):
        assert_rel(k, bwd[k], ob[k])


@pytest.mark.slow
def test_chained_block_and_loss_gpt8b_sampled():
    # full 8.3B shapes: every sampled token's loss, dH and dX depend only on
    # that token's row of the chain
    dev = gpu_or_skip()
    w = wl.WORKLOADS["gpt8b"]
    mi, ci, fwd, ce, bwd, ev, gs = chained(w, dev)
    rows = wl.sample_indices(w.T, 32, seed=0)
    X, A, B, bA, bB = (mi[k].cpu() for k in ("X", "A", "B", "bA", "bB"))
    E, y = ci["E"].cpu(), ci["targets"].cpu().numpy()
    of = oracle.mlp_forward(X[rows], A, bA, B, bB)
    oc = oracle.ce(of["Z"], E, y[rows], w.v_valid, grad_scale=gs, want_dE=False)
    ob = oracle.mlp_backward(X[rows], A, bA, B, oc["dH"], want=("dX",))
    assert_loss("loss", ce["loss"].cpu()[rows], oc["loss"])
    assert torch.equal(ev["loss"], ce["loss"])
    assert_rel("dH", ce["dH"].cpu()[rows], oc["dH"])
    assert_rel("dX", bwd["dX"].cpu()[rows], ob["dX"])
