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
    # widths from 6144 on: dA reads X^T built chunk by chunk, dB reads Y^T with the dZ chunks as B
    "wide_f_x_copy": (512, 256, 6144, 4, "bf16"),
    "wide_h_y_copy": (512, 6144, 512, 4, "bf16"),
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


SWIGLU_SP_CASES = {
    # name: (T, h, f, t, dtype)
    "bf16": (512, 192, 512, 4, "bf16"),
    "f32": (512, 192, 512, 4, "f32"),
    # 2f = 6144: dW1 reads X^T built chunk by chunk; h = 6144: dW2 reads Y^T
    "wide_f_x_copy": (256, 128, 3072, 2, "bf16"),
    "wide_h_y_copy": (256, 6144, 256, 2, "bf16"),
}


@pytest.mark.parametrize("case", list(SWIGLU_SP_CASES))
def test_swiglu_seq_parallel_matches_oracle(case):
    dev = gpu_or_skip()
    T, h, f, t, dtype = SWIGLU_SP_CASES[case]
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


LIN_SP_CASES = {
    # name: (T, n_in, n_out, t, dtype)
    # both partitions valid: n_out / t (column) and n_in / t (row) are whole 64-wide blocks
    "bf16": (512, 512, 256, 4, "bf16"),
    "bf16_wide": (1024, 512, 1024, 8, "bf16"),
    # output width 6144: dW reads the K-major copy of X (made chunk by chunk for the column form)
    "bf16_wide_out": (512, 256, 6144, 4, "bf16"),
    "f32": (256, 128, 256, 2, "f32"),
}


@pytest.mark.parametrize("case", list(LIN_SP_CASES))
def test_linear_seq_parallel_matches_oracle_and_dense(case):
    dev = gpu_or_skip()
    T, n_in, n_out, t, dtype = LIN_SP_CASES[case]
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator().manual_seed(77)
    X = torch.randn(T, n_in, generator=g).to(dt)
    Wc = (0.05 * torch.randn(n_in, n_out, generator=g)).to(dt)     # column-parallel: split n_out
    Wr = (0.05 * torch.randn(n_in, n_out, generator=g)).to(dt)     # row-parallel: split n_in
    b = (0.1 * torch.randn(n_out, generator=g)).float()
    dY = torch.randn(T, n_out, generator=g).to(dt)
    Xd, Wcd, Wrd, bd, dYd = (x.to(dev) for x in (X, Wc, Wr, b, dY))
    rows = T // t
    # column-parallel entry: X (and dX) as chunks
    Yc = tp.tp_column_linear_forward_sp(_split(Xd, t), Wcd, t, bd)
    gc = tp.tp_column_linear_backward_sp(dYd, _split(Xd, t), Wcd, t)
    # row-parallel exit: Y (and dY) as chunks
    Yr = tp.tp_row_linear_forward_sp(Xd, Wrd, t, bd)
    gr = tp.tp_row_linear_backward_sp(_split(dYd, t), Xd, Wrd, t)
    assert tp.device_status() == 0
    assert_rel("column Y", Yc, oracle.linear_forward(X, Wc, b))
    oc = oracle.linear_backward(X, Wc, dY)
    assert_rel("column dX", torch.cat(gc["dX"]), oc["dX"])
    assert_rel("column dW", gc["dW"], oc["dW"])
    assert_rel("column db", gc["db"], oc["db"])
    yr = oracle.linear_forward(X, Wr, b)
    for r in range(t):
        assert_rel(f"row Y[{r}]", Yr[r], yr[r * rows:(r + 1) * rows])
    orr = oracle.linear_backward(X, Wr, dY)
    for k in ("dX", "dW", "db"):
        assert_rel(f"row {k}", gr[k], orr[k])
    # bit for bit the dense calls
    Yc_d = tp.tp_linear_forward(Xd, Wcd, t, "column", bd)
    gc_d = tp.tp_linear_backward(dYd, Xd, Wcd, t, "column")
    Yr_d = tp.tp_linear_forward(Xd, Wrd, t, "row", bd)
    gr_d = tp.tp_linear_backward(dYd, Xd, Wrd, t, "row")
    assert torch.equal(Yc, Yc_d) and torch.equal(torch.cat(Yr), Yr_d)
    assert torch.equal(torch.cat(gc["dX"]), gc_d["dX"])
    for k in ("dW", "db"):
        assert torch.equal(gc[k], gc_d[k]) and torch.equal(gr[k], gr_d[k]), k
    assert torch.equal(gr["dX"], gr_d["dX"])


def test_attention_projections_seq_parallel():
    dev = gpu_or_skip()
    T, h, nq, nkv, d, t = 512, 256, 8, 4, 64, 4
    w = wl.custom("sp_attn", T=T, h=h, f=0, v_valid=0, v_pad=0, t=t, n_heads=nq, n_kv_heads=nkv, head_dim=d)
    ai = wl.attn_inputs(w, seed=0)
    g = {k: v.to(dev) for k, v in ai.items()}
    qkv = tp.tp_attn_qkv_forward_sp(_split(g["X"], t), g["Wqkv"], nq, nkv, d, t, g["bqkv"])
    gq = tp.tp_attn_qkv_backward_sp(g["dQKV"], _split(g["X"], t), g["Wqkv"], nq, nkv, d, t)
    zc = tp.tp_attn_out_forward_sp(g["O"], g["Wo"], nq, d, t, g["bo"])
    go = tp.tp_attn_out_backward_sp(_split(g["dZ"], t), g["O"], g["Wo"], nq, d, t)
    assert tp.device_status() == 0
    assert_rel("QKV", qkv, oracle.linear_forward(ai["X"], ai["Wqkv"], ai["bqkv"]))
    ob = oracle.linear_backward(ai["X"], ai["Wqkv"], ai["dQKV"])
    assert_rel("dX", torch.cat(gq["dX"]), ob["dX"])
    assert_rel("dWqkv", gq["dWqkv"], ob["dW"])
    assert_rel("Z", torch.cat(zc), oracle.linear_forward(ai["O"], ai["Wo"], ai["bo"]))
    oo = oracle.linear_backward(ai["O"], ai["Wo"], ai["dZ"])
    assert_rel("dO", go["dO"], oo["dX"])
    assert_rel("dWo", go["dWo"], oo["dW"])
    assert_rel("dbo", go["dbo"], oo["db"])
    # the dense calls give the same bits
    assert torch.equal(qkv, tp.tp_attn_qkv_forward(g["X"], g["Wqkv"], nq, nkv, d, t, g["bqkv"]))
    assert torch.equal(torch.cat(zc), tp.tp_attn_out_forward(g["O"], g["Wo"], nq, d, t, g["bo"]))
