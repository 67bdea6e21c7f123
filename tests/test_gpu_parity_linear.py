"""GPU parity of the linear primitives (tp_linear_*, column- and
row-parallel) and the attention projections (tp_attn_qkv_*, tp_attn_out_*)
against the fp64 CPU oracle, every output element, through the C ABI.
"""

import pytest
import torch

import oracle
import vocab_ce_gb300 as tp
from vocab_ce_gb300 import workloads as wl
from _parity import assert_rel, gpu_or_skip

pytestmark = pytest.mark.gpu


def _rand(shape, dtype, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (std * torch.randn(*shape, generator=g)).to(dtype)


LINEAR_CASES = {
    # name: (T, n_in, n_out, t, parallel, dtype)
    "column_ragged": (333, 200, 384, 2, "column", "bf16"),
    "row_ragged": (333, 384, 200, 2, "row", "bf16"),
    "column_multi_tile": (700, 512, 1536, 4, "column", "bf16"),
    "row_multi_tile": (700, 1536, 512, 4, "row", "bf16"),
    # n_out >= 6144: dW reads a transposed copy of X (rows padded from 301 to 304 tokens)
    "column_wide_out": (301, 256, 6144, 4, "column", "bf16"),
    "row_wide_out": (301, 512, 6144, 2, "row", "bf16"),
    "column_f32": (130, 96, 256, 4, "column", "f32"),
    "row_f32": (130, 256, 96, 4, "row", "f32"),
}


@pytest.mark.parametrize("case", list(LINEAR_CASES))
def test_linear_matches_oracle(case):
    dev = gpu_or_skip()
    T, n_in, n_out, t, par, dtype = LINEAR_CASES[case]
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    X, W = _rand((T, n_in), dt, 1), _rand((n_in, n_out), dt, 2, 0.05)
    b, dY = _rand((n_out,), torch.float32, 3, 0.1), _rand((T, n_out), dt, 4)
    Y = tp.tp_linear_forward(X.to(dev), W.to(dev), t, par, b.to(dev))
    g = tp.tp_linear_backward(dY.to(dev), X.to(dev), W.to(dev), t, par)
    assert tp.device_status() == 0
    assert_rel("Y", Y, oracle.linear_forward(X, W, b))
    ob = oracle.linear_backward(X, W, dY)
    for k in ("dX", "dW", "db"):
        assert_rel(k, g[k], ob[k])


@pytest.mark.parametrize("par", ["column", "row"])
def test_linear_shard_count_does_not_change_results(par):
    dev = gpu_or_skip()
    X, W, dY = _rand((512, 1024), torch.bfloat16, 5), _rand((1024, 1024), torch.bfloat16, 6, 0.05), \
        _rand((512, 1024), torch.bfloat16, 7)
    X, W, dY = X.to(dev), W.to(dev), dY.to(dev)
    base = None
    for t in (1, 2, 4, 8, 16):
        cur = {"Y": tp.tp_linear_forward(X, W, t, par), **tp.tp_linear_backward(dY, X, W, t, par)}
        assert tp.device_status() == 0
        if base is None:
            base = {k: v.clone() for k, v in cur.items()}
        else:
            for k in base:
                assert torch.equal(base[k], cur[k]), f"t={t}: {k}"


ATTN_CASES = {
    # name: (T, h, n_heads, n_kv_heads, head_dim, t, dtype)
    "gqa_small": (300, 256, 8, 2, 64, 2, "bf16"),
    "gqa_one_kv_per_shard": (260, 512, 16, 4, 64, 4, "bf16"),
    "mha": (200, 384, 6, 6, 64, 3, "bf16"),
    "gqa_f32": (100, 128, 4, 2, 32, 2, "f32"),
}


@pytest.mark.parametrize("case", list(ATTN_CASES))
def test_attention_projections_match_oracle(case):
    dev = gpu_or_skip()
    T, h, nq, nkv, d, t, dtype = ATTN_CASES[case]
    w = wl.custom(case, T=T, h=h, f=0, v_valid=0, v_pad=0, t=t, dtype=dtype, n_heads=nq, n_kv_heads=nkv,
                  head_dim=d)
    ai = wl.attn_inputs(w, seed=0)
    ai["bqkv"] = _rand(ai["bqkv"].shape, torch.float32, 8, 0.1)
    ai["bo"] = _rand(ai["bo"].shape, torch.float32, 9, 0.1)
    g = {k: v.to(dev) for k, v in ai.items()}
    qkv = tp.tp_attn_qkv_forward(g["X"], g["Wqkv"], nq, nkv, d, t, g["bqkv"])
    gq = tp.tp_attn_qkv_backward(g["dQKV"], g["X"], g["Wqkv"], nq, nkv, d, t)
    z = tp.tp_attn_out_forward(g["O"], g["Wo"], nq, d, t, g["bo"])
    go = tp.tp_attn_out_backward(g["dZ"], g["O"], g["Wo"], nq, d, t)
    assert tp.device_status() == 0
    assert_rel("QKV", qkv, oracle.linear_forward(ai["X"], ai["Wqkv"], ai["bqkv"]))
    ob = oracle.linear_backward(ai["X"], ai["Wqkv"], ai["dQKV"])
    assert_rel("dX", gq["dX"], ob["dX"])
    assert_rel("dWqkv", gq["dWqkv"], ob["dW"])
    assert_rel("dbqkv", gq["dbqkv"], ob["db"])
    assert_rel("Z", z, oracle.linear_forward(ai["O"], ai["Wo"], ai["bo"]))
    oo = oracle.linear_backward(ai["O"], ai["Wo"], ai["dZ"])
    assert_rel("dO", go["dO"], oo["dX"])
    assert_rel("dWo", go["dWo"], oo["dW"])
    assert_rel("dbo", go["dbo"], oo["db"])


def test_attention_head_rules_rejected():
    dev = gpu_or_skip()
    X = torch.zeros((4, 256), dtype=torch.bfloat16, device=dev)
    W = torch.zeros((256, (8 + 2 * 2) * 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(tp.TpceError):
        tp.tp_attn_qkv_forward(X, W, 8, 2, 64, 4)   # 2 key/value heads cannot split over 4 shards
    W3 = torch.zeros((256, (8 + 2 * 3) * 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(tp.TpceError):
        tp.tp_attn_qkv_forward(X, W3, 8, 3, 64, 1)  # 8 query heads do not share 3 key/value heads evenly


def test_linear_empty_batch():
    dev = gpu_or_skip()
    X = torch.empty((0, 128), dtype=torch.bfloat16, device=dev)
    W = torch.randn(128, 256, device=dev).bfloat16()
    Y = tp.tp_linear_forward(X, W, 2, "column")
    g = tp.tp_linear_backward(torch.empty((0, 256), dtype=torch.bfloat16, device=dev), X, W, 2, "column")
    assert tp.device_status() == 0
    assert Y.shape == (0, 256)
    assert torch.count_nonzero(g["dW"]).item() == 0 and torch.count_nonzero(g["db"]).item() == 0
