"""The split tail of the CTA-pair GEMM: with 76 clusters (152 SMs), shapes of
80 tiles (one full wave plus 4 tiles) or 640 tiles (8 waves plus 32) make the
GEMMs split their last wave's tiles along K into 2-8 parts whose fp32
partials the last part sums. Checked against the fp64 oracle, for run-to-run
determinism, and against the unsplit run (no workspace) within rounding.
"""

import ctypes

import pytest
import torch

import oracle
import vocab_ce_gb300 as tp
from vocab_ce_gb300._lib import lib
from vocab_ce_gb300 import workloads as wl
from _parity import assert_loss, assert_rel, gpu_or_skip

pytestmark = pytest.mark.gpu


def _biases(n1, n2, seed):
    g = torch.Generator().manual_seed(4000 + seed)
    return (0.1 * torch.randn(n1, generator=g)).float(), (0.1 * torch.randn(n2, generator=g)).float()


def test_mlp_split_tail_matches_oracle_and_is_deterministic():
    # GEMM1 / dY: 8 x 10 = 80 tiles, K = 4096 (64 K blocks) -> 2 parts per
    # tail tile; dB / dA: 160 tiles, K = 2048 -> too short to split
    dev = gpu_or_skip()
    w = wl.custom("split_mlp", T=2048, h=4096, f=2560, v_valid=0, v_pad=0, t=8)
    mi = wl.mlp_inputs(w, seed=0)
    mi["bA"], mi["bB"] = _biases(w.f, w.h, 0)
    g = {k: v.to(dev) for k, v in mi.items()}
    ws = torch.empty(tp.mlp_workspace_bytes(w.T, w.h, w.f, w.t), dtype=torch.uint8, device=dev)

    def run(fws):
        f = tp.tp_mlp_forward(g["X"], g["A"], g["B"], w.t, g["bA"], g["bB"], ws=fws)
        b = tp.tp_mlp_backward(g["dZ"], g["X"], g["A"], g["B"], f["U"], f["Y"], w.t, ws=ws)
        assert tp.device_status() == 0
        return {**{k: f[k].clone() for k in ("U", "Y", "Z")}, **{k: v.clone() for k, v in b.items()}}

    a = run(ws)
    b = run(ws)
    for k in a:
        assert torch.equal(a[k], b[k]), f"{k}: the split tail is not deterministic"
    rows = wl.sample_indices(w.T, 48, seed=0)
    cols = wl.sample_indices(w.f, 24, seed=1)
    of = oracle.mlp_forward(mi["X"][rows], mi["A"], mi["bA"], mi["B"], mi["bB"])
    for k in ("U", "Y", "Z"):
        assert_rel(k, a[k].cpu()[rows], of[k])
    ob = oracle.mlp_backward(mi["X"][rows], mi["A"], mi["bA"], mi["B"], mi["dZ"][rows], want=("dX",))
    assert_rel("dX", a["dX"].cpu()[rows], ob["dX"])
    oc = oracle.mlp_backward_cols(mi["X"], mi["A"], mi["bA"], mi["B"], mi["dZ"], cols)
    assert_rel("dA[:, cols]", a["dA"].cpu()[:, cols], oc["dA"])
    assert_rel("dB[cols, :]", a["dB"].cpu()[cols, :], oc["dB"])
    assert_rel("dbA[cols]", a["dbA"].cpu()[cols], oc["dbA"])
    # the unsplit forward (through the C ABI with no workspace) agrees to
    # rounding, but not bit for bit: the tail tiles were summed in K parts
    f0 = {k: torch.empty_like(a[k]) for k in ("U", "Y", "Z")}

    def p(x):
        return ctypes.c_void_p(x.data_ptr())
    st = lib().tp_mlp_forward(p(g["X"]), p(g["A"]), p(g["bA"]), p(g["B"]), p(g["bB"]), w.T, w.h, w.f, w.t, 0,
                              p(f0["Z"]), p(f0["U"]), p(f0["Y"]), None, 0,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    # (bf16 outputs: a different fp32 summation order may flip the last bit)
    assert_rel("U unsplit", f0["U"], a["U"])
    assert_rel("Z unsplit", f0["Z"], a["Z"])
    assert not torch.equal(f0["U"], a["U"]), "the last wave was not split"


def test_swiglu_split_tail():
    # gated GEMM1: 8 x 10 tiles of 128 output columns, K = 4096 -> 2 parts
    dev = gpu_or_skip()
    w = wl.custom("split_swiglu", T=2048, h=4096, f=1280, v_valid=0, v_pad=0, t=4, act="swiglu")
    si = wl.swiglu_inputs(w, seed=1)
    si["b1"], si["b2"] = _biases(2 * w.f, w.h, 1)
    g = {k: v.to(dev) for k, v in si.items()}
    ws = torch.empty(tp.swiglu_workspace_bytes(w.T, w.h, w.f, w.t), dtype=torch.uint8, device=dev)
    fwd = tp.tp_swiglu_forward(g["X"], g["W1"], g["W2"], w.t, g["b1"], g["b2"], ws=ws)
    bwd = tp.tp_swiglu_backward(g["dZ"], g["X"], g["W1"], g["W2"], fwd["GU"], fwd["Y"], w.t, ws=ws)
    assert tp.device_status() == 0
    rows = wl.sample_indices(w.T, 48, seed=2)
    of = oracle.swiglu_forward(si["X"][rows], si["W1"], si["b1"], si["W2"], si["b2"])
    for k in ("GU", "Y", "Z"):
        assert_rel(k, fwd[k].cpu()[rows], of[k])
    ob = oracle.swiglu_backward(si["X"][rows], si["W1"], si["b1"], si["W2"], si["dZ"][rows], want=("dX",))
    assert_rel("dX", bwd["dX"].cpu()[rows], ob["dX"])


def test_ce_split_tail_all_four_gemms():
    # statistics: 8 x 80 tiles (r = 32, K = 4096: 2 parts); dl: 8 x 40 per
    # chunk (r = 16, 2 parts); dE: 40 x 16 (r = 32, K = 2048: unsplit); dH:
    # 8 x 16 (r = 52: unsplit) -- and with T = 4096, dH of 16 x 10 = 160 tiles
    # (r = 8, K = 10240: 5 parts) stored by the first chunk and reduce-added by
    # the second (test_ce_split_tail_dH)
    dev = gpu_or_skip()
    w = wl.custom("split_ce", T=2048, h=4096, f=0, v_valid=20000, v_pad=20480, t=8)
    ci = wl.ce_inputs(w, seed=3)
    g = {k: v.to(dev) for k, v in ci.items()}
    gs = 1.0 / w.T
    out = tp.vocab_parallel_ce(g["H"], g["E"], g["targets"], w.v_valid, w.t, grad_scale=gs)
    again = tp.vocab_parallel_ce(g["H"], g["E"], g["targets"], w.v_valid, w.t, grad_scale=gs)
    assert tp.device_status() == 0
    for k in out:
        assert torch.equal(out[k], again[k]), f"{k}: the split tail is not deterministic"
    rows = wl.sample_indices(w.T, 32, seed=4)
    ref = oracle.ce(ci["H"][rows], ci["E"], ci["targets"].numpy()[rows], w.v_valid, grad_scale=gs, want_dE=False)
    assert_loss("loss", out["loss"].cpu()[rows], ref["loss"])
    assert_loss("lse", out["lse"].cpu()[rows], ref["lse"])
    assert_rel("dH", out["dH"].cpu()[rows], ref["dH"])
    sub = tp.vocab_parallel_ce(g["H"][:64].contiguous(), g["E"], g["targets"][:64].contiguous(), w.v_valid, w.t)
    ref2 = oracle.ce(ci["H"][:64], ci["E"], ci["targets"].numpy()[:64], w.v_valid)
    assert_rel("dE (64 tokens)", sub["dE"], ref2["dE"])
    assert torch.count_nonzero(out["dE"][w.v_valid:]).item() == 0


def test_ce_split_tail_dH():
    # dH: 16 x 10 = 160 tiles (r = 8), K = one 4-shard chunk of 10,240 ids
    # (160 K blocks) -> 5 parts; chunk 0 stores, chunk 1 reduce-adds
    dev = gpu_or_skip()
    w = wl.custom("split_dh", T=4096, h=2560, f=0, v_valid=20000, v_pad=20480, t=8)
    ci = wl.ce_inputs(w, seed=5)
    g = {k: v.to(dev) for k, v in ci.items()}
    out = tp.vocab_parallel_ce(g["H"], g["E"], g["targets"], w.v_valid, w.t, grad_scale=1.0 / w.T, want_dE=False)
    again = tp.vocab_parallel_ce(g["H"], g["E"], g["targets"], w.v_valid, w.t, grad_scale=1.0 / w.T, want_dE=False)
    assert tp.device_status() == 0
    assert torch.equal(out["dH"], again["dH"])
    rows = wl.sample_indices(w.T, 32, seed=6)
    ref = oracle.ce(ci["H"][rows], ci["E"], ci["targets"].numpy()[rows], w.v_valid, grad_scale=1.0 / w.T,
                    want_dE=False)
    assert_loss("loss", out["loss"].cpu()[rows], ref["loss"])
    assert_rel("dH", out["dH"].cpu()[rows], ref["dH"])
