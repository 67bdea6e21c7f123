"""The path captured into a CUDA graph: one eager call of each entry point
(which loads the kernels and sets their attributes), then the MLP block
forward/backward and the fused CE forward/backward captured into one graph
with preallocated outputs and workspaces, and replayed. Replays must give
the eager results bit for bit, and must read the input buffers afresh.
"""

import pytest
import torch

import vocab_ce_gb300 as tp
from vocab_ce_gb300 import workloads as wl
from _parity import gpu_or_skip

pytestmark = pytest.mark.gpu


def test_block_and_loss_replay_from_a_cuda_graph():
    dev = gpu_or_skip()
    w = wl.custom("graph", T=512, h=256, f=1024, v_valid=1900, v_pad=2048, t=4)
    mi = wl.mlp_inputs(w, seed=0, device=dev)
    ci = wl.ce_inputs(w, seed=0, device=dev)
    T, h, f = w.T, w.h, w.f
    bf = torch.bfloat16
    fo = {"Z": torch.empty((T, h), dtype=bf, device=dev), "U": torch.empty((T, f), dtype=bf, device=dev),
          "Y": torch.empty((T, f), dtype=bf, device=dev)}
    bo = {"dX": torch.empty((T, h), dtype=bf, device=dev), "dA": torch.empty((h, f), dtype=bf, device=dev),
          "dB": torch.empty((f, h), dtype=bf, device=dev), "dbA": torch.empty(f, device=dev),
          "dbB": torch.empty(h, device=dev)}
    co = {"loss": torch.empty(T, device=dev), "lse": torch.empty(T, device=dev),
          "dH": torch.empty((T, h), dtype=bf, device=dev), "dE": torch.empty((w.v_pad, h), dtype=bf, device=dev)}
    mws = torch.empty(tp.mlp_workspace_bytes(T, h, f, w.t), dtype=torch.uint8, device=dev)
    cws = torch.empty(tp.ce_workspace_bytes(T, h, w.v_pad, w.t), dtype=torch.uint8, device=dev)

    def step():
        tp.tp_mlp_forward(mi["X"], mi["A"], mi["B"], w.t, mi["bA"], mi["bB"], out=fo, ws=mws)
        tp.tp_mlp_backward(mi["dZ"], mi["X"], mi["A"], mi["B"], fo["U"], fo["Y"], w.t, out=bo, ws=mws)
        tp.vocab_parallel_ce(ci["H"], ci["E"], ci["targets"], w.v_valid, w.t, grad_scale=1.0 / T, out=co, ws=cws)

    def snapshot():
        return {k: v.clone() for d in (fo, bo, co) for k, v in d.items()}

    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # eager: loads the kernels, sets their attributes
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert tp.device_status() == 0
    ref = snapshot()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for k in fo:
        fo[k].zero_()
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        assert tp.device_status() == 0
        cur = snapshot()
        for k in ref:
            assert torch.equal(cur[k], ref[k]), k

    # new input values in the same buffers: the replay reads them
    mi["X"].copy_(torch.flip(mi["X"], dims=[0]))
    ci["H"].copy_(torch.flip(ci["H"], dims=[0]))
    g.replay()
    torch.cuda.synchronize()
    replayed = snapshot()
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager = snapshot()
    for k in eager:
        assert torch.equal(replayed[k], eager[k]), k
    assert not torch.equal(replayed["Z"], ref["Z"])
