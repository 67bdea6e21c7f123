"""GPU parity of the sequence-parallel entry/exit ("Mathematical Foundations
of Megatron-LM 1D Slicing", section "Sequence Parallelism"): X, Z, dZ and dX
as t sequence-chunk buffers. Compared with the oracle's sequence-parallel
restatement (all-gather of the X chunks, reduce-scatter of the shard partials
into Z chunks) and, bit for bit, with the dense calls on the gathered tensors.
"""

import pytest
import torch

import oracle
import vocab_ce_gb300 as tp
from vocab_ce_gb300 import workloads as wl
from _parity import assert_rel, gpu_or_skip

pytestmark = pytest.mark.gpu


def _biases(n1, n2, seed):
    g = torch.Generator().manual_seed(3000 + seed)
    return (0.1 * torch.randn(n1, generator=g)).float(), (0.1 * torch.randn(n2, generator=g)).float()


def _split(x, t):
    rows = x.shape[0] // t
    return [x[i * rows:(i + 1) * rows].contiguous() for i in range(t)]


SP_CASES = {
    # name: (T, h, f, t, dtype)
    "four_chunks": (512, 256, 1024, 4, "bf16"),
    "chunk_inside_pair_tile": (768, 200, 384, 2, "bf16"),     # 384-row chunks: a 256-row pair tile spans two
    "ragged_last_pair_tile": (640, 136, 640, 5, "bf16"),      # T/128 odd: the last tile's second CTA is past T
    "sixteen_chunks": (2048, 128, 1024, 16, "bf16"),
    "fp32": (256, 128, 256, 2, "f32"),
}


@pytest.mark.parametrize("case", list(SP_CASES))
def test_mlp_seq_parallel_matches_oracle(case):
    dev = gpu_or_skip()
    T, h, f, t, dtype = SP_CASES[case]
    w = wl.custom(case, T=T, h=h, f=f, v_valid=0, v_pad=0, t=t, dtype=dtype)
    mi = wl.mlp_inputs(w, seed=0)
    mi["bA"], mi["bB"] = _biases(f, h, 0)
    g = {k: v.to(dev) for k, v in mi.items()}
    Xc, dZc = _split(g["X"], t), _split(g["dZ"], t)
    fwd = tp.tp_mlp_forward_sp(Xc, g["A"], g["B"], t, g["bA"], g["bB"])
    bwd = tp.tp_mlp_backward_sp(dZc, Xc, g["A"], g["B"], fwd["U"], fwd["Y"], t)
    assert tp.device_status() == 0
    ref = oracle.mlp_seq_parallel(_split(mi["X"], t), mi["A"], mi["bA"], mi["B"], mi["bB"], _split(mi["dZ"], t))
    for r in range(t):
        assert_rel(f"Z[{r}]", fwd["Z"][r], ref["Z"][r])
        assert_rel(f"dX[{r}]", bwd["dX"][r], ref["dX"][r])
    assert_rel("dA", bwd["dA"], ref["dA"])
    assert_rel("dB", bwd["dB"], ref["dB"])
    assert_rel("dbB", bwd["dbB"], oracle.bias_grad(mi["dZ"]))
    # the same arithmetic as the dense calls on the gathered tensors, bit for bit
    dfw = tp.tp_mlp_forward(g["X"], g["A"], g["B"], t, g["bA"], g["bB"])
    dbw = tp.tp_mlp_backward(g["dZ"], g["X"], g["A"], g["B"], dfw["U"], dfw["Y"], t)
    assert tp.device_status() == 0
    assert torch.equal(torch.cat(fwd["Z"]), dfw["Z"])
    assert torch.equal(fwd["U"], dfw["U"]) and torch.equal(fwd["Y"], dfw["Y"])
    assert torch.equal(torch.cat(bwd["dX"]), dbw["dX"])
    for k in ("dA", "dB", "dbA", "dbB"):
        assert torch.equal(bwd[k], dbw[k]), k


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_swiglu_seq_parallel_matches_oracle(dtype):
    dev = gpu_or_skip()
    T, h, f, t = 512, 192, 512, 4
    w = wl.custom("sp_swiglu", T=T, h=h, f=f, v_valid=0, v_pad=0, t=t, dtype=dtype, act="swiglu")
    si = wl.swiglu_inputs(w, seed=0)
    si["b1"], si["b2"] = _biases(2 * f, h, 1)
    g = {k: v.to(dev) for k, v in si.items()}
    Xc, dZc = _split(g["X"], t), _split(g["dZ"], t)
    fwd = tp.tp_swiglu_forward_sp(Xc, g["W1"], g["W2"], t, g["b1"], g["b2"])
    bwd = tp.tp_swiglu_backward_sp(dZc, Xc, g["W1"], g["W2"], fwd["GU"], fwd["Y"], t)
    assert tp.device_status() == 0
    of = oracle.swiglu_forward(si["X"], si["W1"], si["b1"], si["W2"], si["b2"])
    ob = oracle.swiglu_backward(si["X"], si["W1"], si["b1"], si["W2"], si["dZ"])
    rows = T // t
    for r in range(t):
        assert_rel(f"Z[{r}]", fwd["Z"][r], of["Z"][r * rows:(r + 1) * rows])
        assert_rel(f"dX[{r}]", bwd["dX"][r], ob["dX"][r * rows:(r + 1) * rows])
    for k in ("dW1", "dW2", "db1", "db2"):
        assert_rel(k, bwd[k], ob[k])
    dfw = tp.tp_swiglu_forward(g["X"], g["W1"], g["W2"], t, g["b1"], g["b2"])
    dbw = tp.tp_swiglu_backward(g["dZ"], g["X"], g["W1"], g["W2"], dfw["GU"], dfw["Y"], t)
    assert torch.equal(torch.cat(fwd["Z"]), dfw["Z"])
    assert torch.equal(torch.cat(bwd["dX"]), dbw["dX"])
    for k in ("dW1", "dW2", "db1", "db2"):
        assert torch.equal(bwd[k], dbw[k]), k


def test_seq_parallel_chunks_are_separate_buffers():
    # the chunks need not be adjacent in memory: give them gaps and a shuffled
    # allocation order, and check the result is unchanged
    dev = gpu_or_skip()
    T, h, f, t = 512, 128, 512, 4
    w = wl.custom("sp_gaps", T=T, h=h, f=f, v_valid=0, v_pad=0, t=t)
    mi = wl.mlp_inputs(w, seed=2)
    g = {k: v.to(dev) for k, v in mi.items()}
    rows = T // t
    pool = torch.zeros((3 * T, h), dtype=torch.bfloat16, device=dev)
    order = [2, 0, 3, 1]
    Xc = [pool[(2 * order[i] + 1) * rows:(2 * order[i] + 2) * rows] for i in range(t)]
    for i in range(t):
        Xc[i].copy_(g["X"][i * rows:(i + 1) * rows])
    out_pool = torch.full((3 * T, h), 7.0, dtype=torch.bfloat16, device=dev)
    Zc = [out_pool[(2 * order[i]) * rows:(2 * order[i] + 1) * rows] for i in range(t)]
    fwd = tp.tp_mlp_forward_sp(Xc, g["A"], g["B"], t, out={"Z": Zc})
    dense = tp.tp_mlp_forward(g["X"], g["A"], g["B"], t)
    assert tp.device_status() == 0
    assert torch.equal(torch.cat(fwd["Z"]), dense["Z"])
    # the rows between the chunks were not touched
    for i in range(t):
        gap = out_pool[(2 * order[i] + 1) * rows:(2 * order[i] + 2) * rows]
        assert torch.all(gap == 7.0)
