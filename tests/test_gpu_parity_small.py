"""GPU parity, small and medium sizes: every output element compared with the
fp64 CPU oracle on the same seeded inputs, through the C ABI.

Cases span several tiles in every dimension and ragged tails (T, h, N not
multiples of the 128 x 256 tile; vocabulary shards that are odd multiples of
128; shards made only of padded ids).
"""

import numpy as np
import pytest
import torch

import oracle
import vocab_ce_gb300 as tp
from vocab_ce_gb300 import workloads as wl
from _parity import assert_loss, assert_rel, gpu_or_skip

pytestmark = pytest.mark.gpu


def _biases(w, seed):
    g = torch.Generator().manual_seed(1000 + seed)
    return (0.1 * torch.randn(w.f, generator=g)).float(), (0.1 * torch.randn(w.h, generator=g)).float()


def run_mlp(w, dev, seed=0, nonzero_bias=True):
    mi = wl.mlp_inputs(w, seed=seed)
    if nonzero_bias:
        mi["bA"], mi["bB"] = _biases(w, seed)
    g = {k: v.to(dev) for k, v in mi.items()}
    fwd = tp.tp_mlp_forward(g["X"], g["A"], g["B"], w.t, g["bA"], g["bB"])
    bwd = tp.tp_mlp_backward(g["dZ"], g["X"], g["A"], g["B"], fwd["U"], fwd["Y"], w.t)
    assert tp.device_status() == 0
    return mi, fwd, bwd


MLP_CASES = {
    # name: (T, h, f, t, dtype)
    "tiny_shape_bf16": (32, 64, 256, 2, "bf16"),
    "ragged": (333, 200, 384, 2, "bf16"),
    "multi_tile": (640, 512, 1024, 4, "bf16"),
    "one_token": (1, 64, 128, 2, "bf16"),
    "min_hidden": (5, 8, 128, 2, "bf16"),            # h = 8: one k-block, mostly zero-filled by TMA
    "min_hidden_f32": (5, 8, 128, 2, "f32"),
    "wide_n_tiles": (1000, 1536, 3072, 8, "bf16"),   # picks 192-wide tiles
    "ragged_f32": (333, 200, 384, 2, "f32"),
    "multi_tile_f32": (300, 256, 512, 4, "f32"),
}


def test_tiny_config_fp32_matches_oracle():
    # the tiny workload as specified: fp32 tensors (tf32 tensor-core path), t = 2
    dev = gpu_or_skip()
    w = wl.WORKLOADS["tiny"]
    assert w.dtype == "f32"
    mi, fwd, bwd = run_mlp(w, dev)
    assert fwd["Z"].dtype == torch.float32
    of = oracle.mlp_forward(mi["X"], mi["A"], mi["bA"], mi["B"], mi["bB"])
    ob = oracle.mlp_backward(mi["X"], mi["A"], mi["bA"], mi["B"], mi["dZ"])
    for k in ("U", "Y", "Z"):
        assert_rel(k, fwd[k], of[k])
    for k in ("dX", "dA", "dB", "dbA", "dbB"):
        assert_rel(k, bwd[k], ob[k])
    ci = wl.ce_inputs(w, seed=0)
    g = {k: v.to(dev) for k, v in ci.items()}
    out = tp.vocab_parallel_ce(g["H"], g["E"], g["targets"], w.v_valid, w.t, grad_scale=1.0)
    assert tp.device_status() == 0
    ref = oracle.ce(ci["H"], ci["E"], ci["targets"].numpy(), w.v_valid, grad_scale=1.0)
    assert_loss("loss", out["loss"], ref["loss"])
    assert_rel("dH", out["dH"], ref["dH"])
    assert_rel("dE", out["dE"], ref["dE"])


def test_gelu_and_derivative_evaluation_error_fp32():
    # GeLU and GeLU' on the device (erf by Abramowitz & Stegun 7.1.26, error
    # <= 1.5e-7) checked at their own accuracy through the fp32 API: with
    # A = B = I, bA = 0 and dZ = 1, a single token gives U = tf32(X), Y =
    # GeLU(U) and dbA = dY (.) GeLU'(U) = GeLU'(U) exactly up to the device
    # evaluation of the two functions.
    dev = gpu_or_skip()
    h = f = 256
    X = torch.linspace(-7.0, 7.0, h, dtype=torch.float32).reshape(1, h).to(dev)
    I = torch.eye(h, dtype=torch.float32, device=dev)
    fwd = tp.tp_mlp_forward(X, I, I, 2)
    bwd = tp.tp_mlp_backward(torch.ones(1, h, device=dev), X, I, I, fwd["U"], fwd["Y"], 2)
    assert tp.device_status() == 0
    U = fwd["U"].double().cpu().numpy()[0]
    Y = fwd["Y"].double().cpu().numpy()[0]
    dU = bwd["dbA"].double().cpu().numpy()
    gelu = np.array([oracle.gelu(u) for u in U])
    dgelu = np.array([oracle.gelu_grad(u) for u in U])
    assert np.abs(Y - gelu).max() <= 1e-6 * max(1.0, np.abs(U).max())
    assert np.abs(dU - dgelu).max() <= 1e-6


def test_gelu_far_tails_fp32():
    # |u| up to 120: e^{-u^2/2} underflows to 0, and GeLU -> max(u, 0),
    # GeLU' -> 1 or 0, with no NaN
    dev = gpu_or_skip()
    h = f = 256
    X = torch.linspace(-120.0, 120.0, h, dtype=torch.float32).reshape(1, h).to(dev)
    I = torch.eye(h, dtype=torch.float32, device=dev)
    fwd = tp.tp_mlp_forward(X, I, I, 2)
    bwd = tp.tp_mlp_backward(torch.ones(1, h, device=dev), X, I, I, fwd["U"], fwd["Y"], 2)
    assert tp.device_status() == 0
    U = fwd["U"].double().cpu().numpy()[0]
    Y = fwd["Y"].double().cpu().numpy()[0]
    dU = bwd["dbA"].double().cpu().numpy()
    assert np.isfinite(Y).all() and np.isfinite(dU).all()
    gelu = np.array([oracle.gelu(u) for u in U])
    dgelu = np.array([oracle.gelu_grad(u) for u in U])
    assert np.abs(Y - gelu).max() <= 1e-6 * np.abs(U).max()
    assert np.abs(dU - dgelu).max() <= 1e-6


@pytest.mark.parametrize("case", list(MLP_CASES))
def test_mlp_matches_oracle(case):
    dev = gpu_or_skip()
    T, h, f, t, dtype = MLP_CASES[case]
    w = wl.custom(case, T=T, h=h, f=f, v_valid=0, v_pad=0, t=t, dtype=dtype)
    mi, fwd, bwd = run_mlp(w, dev)
    of = oracle.mlp_forward(mi["X"], mi["A"], mi["bA"], mi["B"], mi["bB"])
    ob = oracle.mlp_backward(mi["X"], mi["A"], mi["bA"], mi["B"], mi["dZ"])
    for k in ("U", "Y", "Z"):
        assert_rel(k, fwd[k], of[k])
    for k in ("dX", "dA", "dB", "dbA", "dbB"):
        assert_rel(k, bwd[k], ob[k])


def test_mlp_shard_count_does_not_change_results():
    # Z = sum_i Y_i B_i equals the unsharded product for every t; on one GPU the
    # shards are tile coordinates, so the results agree bit for bit.
    dev = gpu_or_skip()
    base = None
    for t in (1, 2, 4, 8, 16):
        w = wl.custom(f"t{t}", T=512, h=256, f=1024, v_valid=0, v_pad=0, t=t)
        mi, fwd, bwd = run_mlp(w, dev)
        cur = {**{k: fwd[k].cpu() for k in ("Z", "Y")}, **{k: v.cpu() for k, v in bwd.items()}}
        if base is None:
            base = cur
            of = oracle.mlp_forward(mi["X"], mi["A"], mi["bA"], mi["B"], mi["bB"])
            ob = oracle.mlp_backward(mi["X"], mi["A"], mi["bA"], mi["B"], mi["dZ"])
            assert_rel("Z", fwd["Z"], of["Z"])
            assert_rel("dX", bwd["dX"], ob["dX"])
        else:
            for k in base:
                assert torch.equal(base[k], cur[k]), f"t={t}: {k} differs from t=1"


CE_CASES = {
    # name: (T, h, v_pad, v_valid, t, dtype)
    "tiny_shape_bf16": (32, 64, 512, 512, 2, "bf16"),
    "ragged_bn128": (333, 200, 768, 700, 2, "bf16"),          # shard = 384 ids: 128-wide tiles
    "padded_shards": (130, 96, 2048, 1800, 16, "bf16"),       # shard 15 holds only padding
    "single_shard": (257, 128, 1024, 1000, 1, "bf16"),        # t = 1: the unsharded loss
    "min_hidden": (7, 8, 256, 200, 2, "bf16"),                # h = 8: one mostly zero-filled k-block
    "multi_tile": (600, 320, 4096, 4000, 4, "bf16"),
    "wide_h": (700, 1536, 3072, 3000, 4, "bf16"),             # dE / dH pick 192-wide tiles
    # 25 row-blocks x 4 shards: each shard's 6 tiles are cut into 3 runs of 2
    # (300 work units, 4 waves over the CTA pairs), so the combine folds 3
    # partial statistics per shard
    "runs_split_shards": (6400, 64, 6144, 6000, 4, "bf16"),
    # h >= 6144: dE reads a transposed copy of dl (rows padded from 300 to 304 tokens)
    "wide_h_transposed_dl": (300, 6144, 1024, 1000, 4, "bf16"),
    "ragged_f32": (333, 200, 768, 700, 2, "f32"),
    "padded_shards_f32": (130, 96, 2048, 1800, 16, "f32"),
}


@pytest.mark.parametrize("case", list(CE_CASES))
def test_ce_matches_oracle(case):
    dev = gpu_or_skip()
    T, h, v_pad, v_valid, t, dtype = CE_CASES[case]
    assert tp.pad_vocab(v_valid, t) <= v_pad
    w = wl.custom(case, T=T, h=h, f=0, v_valid=v_valid, v_pad=v_pad, t=t, dtype=dtype)
    ci = wl.ce_inputs(w, seed=0)
    ci["targets"][0] = 0
    ci["targets"][-1] = v_valid - 1
    g = {k: v.to(dev) for k, v in ci.items()}
    gs = 1.0 / T
    out = tp.vocab_parallel_ce(g["H"], g["E"], g["targets"], v_valid, t, grad_scale=gs)
    assert tp.device_status() == 0
    ref = oracle.ce(ci["H"], ci["E"], ci["targets"].numpy(), v_valid, grad_scale=gs)
    assert_loss("loss", out["loss"], ref["loss"])
    assert_loss("lse", out["lse"], ref["lse"])
    assert_rel("dH", out["dH"], ref["dH"])
    assert_rel("dE", out["dE"], ref["dE"])
    # padded vocabulary rows get exactly zero gradient
    assert torch.count_nonzero(out["dE"][v_valid:]).item() == 0
    # the sharded statistics restatement of the oracle agrees with the loss too
    sh = oracle.ce_sharded(ci["H"], ci["E"], ci["targets"].numpy(), v_valid, t)
    assert_loss("loss vs sharded oracle", out["loss"], sh["loss"])


@pytest.mark.parametrize("gs,dtype", [(0.0, "bf16"), (-0.75, "bf16"), (1.0e4, "bf16"), (-0.75, "f32")])
def test_ce_grad_scale_zero_negative_and_large(gs, dtype):
    # The dl epilogue folds a positive grad_scale into the exponent,
    # exp(l - (lse - ln g)), and multiplies by it otherwise: a zero scale gives
    # zero gradients, a negative one flips their sign, a large one stays finite.
    dev = gpu_or_skip()
    T, h, v_pad, v_valid, t = 200, 128, 1024, 1000, 4
    w = wl.custom("grad_scale", T=T, h=h, f=0, v_valid=v_valid, v_pad=v_pad, t=t, dtype=dtype)
    ci = wl.ce_inputs(w, seed=3)
    g = {k: v.to(dev) for k, v in ci.items()}
    out = tp.vocab_parallel_ce(g["H"], g["E"], g["targets"], v_valid, t, grad_scale=gs)
    assert tp.device_status() == 0
    ref = oracle.ce(ci["H"], ci["E"], ci["targets"].numpy(), v_valid, grad_scale=gs)
    assert_loss("loss", out["loss"], ref["loss"])
    if gs == 0.0:
        assert torch.count_nonzero(out["dH"]).item() == 0 and torch.count_nonzero(out["dE"]).item() == 0
    else:
        assert_rel(f"dH (grad_scale {gs}, {dtype})", out["dH"], ref["dH"])
        assert_rel(f"dE (grad_scale {gs}, {dtype})", out["dE"], ref["dE"])


def test_ce_backward_with_shards_split_into_chunks():
    # The dl scratch of one vocabulary chunk is bounded (1 GiB): at 66,000
    # tokens one 8,192-id shard alone would need 1.08 GB, so each shard is cut
    # into two 4,096-id chunks and dH adds four chunks in fp32. Every output
    # against the oracle (h = 16 keeps the oracle's full softmax to seconds).
    dev = gpu_or_skip()
    T, h, v_pad, v_valid, t = 66000, 16, 16384, 16000, 2
    w = wl.custom("split_shards", T=T, h=h, f=0, v_valid=v_valid, v_pad=v_pad, t=t)
    ci = wl.ce_inputs(w, seed=4)
    g = {k: v.to(dev) for k, v in ci.items()}
    out = tp.vocab_parallel_ce(g["H"], g["E"], g["targets"], v_valid, t, grad_scale=1.0 / T)
    assert tp.device_status() == 0
    ref = oracle.ce(ci["H"], ci["E"], ci["targets"].numpy(), v_valid, grad_scale=1.0 / T)
    assert_loss("loss", out["loss"], ref["loss"])
    assert_rel("dH", out["dH"], ref["dH"])
    assert_rel("dE", out["dE"], ref["dE"])
    assert torch.count_nonzero(out["dE"][v_valid:]).item() == 0


def test_ce_partial_statistics_fold_is_repeatable_on_a_dirty_workspace():
    # A shard cut into several runs has its partial (max, sumexp) pairs folded
    # by the epilogue that draws the last ticket. The tickets live in the
    # caller's workspace, which may hold anything: each call clears them.
    # Two calls on a workspace filled with 0xff bytes, then a third after a
    # call of another shape, give the same losses bit for bit, matching the
    # oracle.
    dev = gpu_or_skip()
    T, h, v_pad, v_valid, t, _ = CE_CASES["runs_split_shards"]
    w = wl.custom("fold", T=T, h=h, f=0, v_valid=v_valid, v_pad=v_pad, t=t)
    ci = wl.ce_inputs(w, seed=3)
    g = {k: v.to(dev) for k, v in ci.items()}
    nbytes = tp.ce_workspace_bytes(T, h, v_pad, t, grads=False)
    ws = torch.full((nbytes,), 255, dtype=torch.uint8, device=dev)
    runs = []
    for _ in range(2):
        out = tp.vocab_parallel_ce(g["H"], g["E"], g["targets"], v_valid, t, grads=False, ws=ws)
        assert tp.device_status() == 0
        runs.append(out["loss"].clone())
    # a call of another shape through the same workspace, then the first again
    w2 = wl.custom("fold2", T=1000, h=h, f=0, v_valid=3900, v_pad=4096, t=8)
    c2 = {k: v.to(dev) for k, v in wl.ce_inputs(w2, seed=4).items()}
    ws.fill_(255)
    tp.vocab_parallel_ce(c2["H"], c2["E"], c2["targets"], 3900, 8, grads=False, ws=ws)
    out = tp.vocab_parallel_ce(g["H"], g["E"], g["targets"], v_valid, t, grads=False, ws=ws)
    assert tp.device_status() == 0
    runs.append(out["loss"].clone())
    assert torch.equal(runs[0], runs[1]) and torch.equal(runs[0], runs[2])
    ref = oracle.ce(ci["H"], ci["E"], ci["targets"].numpy(), v_valid, grads=False)
    assert_loss("loss after the fold", runs[2], ref["loss"])


def test_ce_forward_only_and_single_gradients():
    dev = gpu_or_skip()
    T, h, v_pad, v_valid, t = 200, 128, 1024, 1000, 4
    w = wl.custom("fo", T=T, h=h, f=0, v_valid=v_valid, v_pad=v_pad, t=t)
    ci = wl.ce_inputs(w, seed=3)
    g = {k: v.to(dev) for k, v in ci.items()}
    ref = oracle.ce(ci["H"], ci["E"], ci["targets"].numpy(), v_valid, grad_scale=1.0)
    fo = tp.vocab_parallel_ce(g["H"], g["E"], g["targets"], v_valid, t, grads=False)
    assert "dH" not in fo and "dE" not in fo
    assert_loss("loss", fo["loss"], ref["loss"])
    only_dh = tp.vocab_parallel_ce(g["H"], g["E"], g["targets"], v_valid, t, want_dE=False)
    assert_rel("dH", only_dh["dH"], ref["dH"])
    only_de = tp.vocab_parallel_ce(g["H"], g["E"], g["targets"], v_valid, t, want_dH=False)
    assert_rel("dE", only_de["dE"], ref["dE"])
    assert tp.device_status() == 0


def test_ce_closed_form_zero_embedding():
    # E = 0 on the real ids: loss = ln(v_valid) for every token, dH = 0
    dev = gpu_or_skip()
    T, h, v_pad, v_valid, t = 256, 64, 2048, 2000, 8
    H = torch.randn(T, h).to(torch.bfloat16).to(dev)
    E = torch.zeros(v_pad, h, dtype=torch.bfloat16, device=dev)
    E[v_valid:] = 3.0  # padded rows must not enter
    y = torch.randint(0, v_valid, (T,), dtype=torch.int32, device=dev)
    out = tp.vocab_parallel_ce(H, E, y, v_valid, t)
    assert tp.device_status() == 0
    assert_loss("loss", out["loss"], np.full(T, np.log(v_valid)))
    assert torch.count_nonzero(out["dH"]).item() == 0


def test_ce_large_logits():
    # logits with standard deviation ~30 (maxima near 100): exp without the running
    # max would overflow fp32; loss, lse and gradients still match the fp64 oracle
    dev = gpu_or_skip()
    T, h, v_pad, v_valid, t = 96, 64, 1024, 1000, 4
    g = torch.Generator().manual_seed(23)
    H = torch.randn(T, h, generator=g).to(torch.bfloat16)
    E = (3.75 * torch.randn(v_pad, h, generator=g)).to(torch.bfloat16)
    y = torch.randint(0, v_valid, (T,), generator=g, dtype=torch.int64).to(torch.int32)
    out = tp.vocab_parallel_ce(H.to(dev), E.to(dev), y.to(dev), v_valid, t, grad_scale=1.0 / T)
    assert tp.device_status() == 0
    assert torch.isfinite(out["loss"]).all() and torch.isfinite(out["dH"].float()).all()
    ref = oracle.ce(H, E, y.numpy(), v_valid, grad_scale=1.0 / T)
    assert float(np.abs(ref["lse"]).max()) > 60.0  # the case really has large logits
    assert_loss("loss", out["loss"], ref["loss"])
    assert_loss("lse", out["lse"], ref["lse"])
    assert_rel("dH", out["dH"], ref["dH"])
    assert_rel("dE", out["dE"], ref["dE"])


def test_ce_single_real_id():
    # v_valid = 1: the softmax over the one real id is exactly the one-hot target,
    # so the loss is 0 and dl, dH, dE vanish exactly; shard 1 holds only padding
    dev = gpu_or_skip()
    T, h, v_pad, v_valid, t = 96, 64, 256, 1, 2
    g = torch.Generator().manual_seed(21)
    H = torch.randn(T, h, generator=g).to(torch.bfloat16).to(dev)
    E = (0.5 * torch.randn(v_pad, h, generator=g)).to(torch.bfloat16).to(dev)
    y = torch.zeros(T, dtype=torch.int32, device=dev)
    out = tp.vocab_parallel_ce(H, E, y, v_valid, t)
    assert tp.device_status() == 0
    assert torch.count_nonzero(out["loss"]).item() == 0
    assert torch.count_nonzero(out["dH"]).item() == 0
    assert torch.count_nonzero(out["dE"]).item() == 0
    # lse is the target logit itself
    ref = oracle.ce(H.cpu(), E.cpu(), y.cpu().numpy(), v_valid, want_dE=False)
    assert_loss("lse", out["lse"], ref["lse"])


def test_empty_token_batch():
    dev = gpu_or_skip()
    h, f, t = 64, 256, 2
    X = torch.empty(0, h, dtype=torch.bfloat16, device=dev)
    A = torch.randn(h, f, device=dev).to(torch.bfloat16)
    B = torch.randn(f, h, device=dev).to(torch.bfloat16)
    fwd = tp.tp_mlp_forward(X, A, B, t)
    assert fwd["Z"].shape == (0, h)
    bwd = tp.tp_mlp_backward(X, X, A, B, fwd["U"], fwd["Y"], t)
    assert torch.count_nonzero(bwd["dA"]).item() == 0 and torch.count_nonzero(bwd["dB"]).item() == 0
    assert torch.count_nonzero(bwd["dbA"]).item() == 0
    E = torch.randn(512, h, device=dev).to(torch.bfloat16)
    ce = tp.vocab_parallel_ce(X, E, torch.empty(0, dtype=torch.int32, device=dev), 500, 2)
    assert ce["loss"].numel() == 0 and torch.count_nonzero(ce["dE"]).item() == 0
    assert tp.device_status() == 0


def test_out_of_range_target_is_reported():
    dev = gpu_or_skip()
    T, h, v_pad, v_valid, t = 64, 64, 512, 500, 2
    H = torch.randn(T, h, device=dev).to(torch.bfloat16)
    E = torch.randn(v_pad, h, device=dev).to(torch.bfloat16)
    y = torch.randint(0, v_valid, (T,), dtype=torch.int32, device=dev)
    y[5] = v_valid  # a padded id is not a valid target
    out = tp.vocab_parallel_ce(H, E, y, v_valid, t, grads=False)
    assert tp.device_status() == 1  # TPCE_ERR_INVALID, then cleared
    loss = out["loss"].cpu()
    assert torch.isnan(loss[5]) and torch.isfinite(loss[:5]).all()
    assert tp.device_status() == 0
