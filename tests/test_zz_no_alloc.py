"""vocab_parallel_ce_loss_static: the fused cross-entropy forward for callers
that cannot allocate device memory (a plugin under a host framework's memory
planner, a latency-critical path that must avoid cudaMalloc's implicit
synchronisation). It takes no workspace: its scratch is a static device array
inside the library.

The GPU test calls it through the C ABI on two calls in a row, each into
caller-owned output buffers allocated before the call, and compares the
losses and log-sum-exps with those of vocab_parallel_ce (the workspace
version) on the same inputs, within the loss tolerance of the parity tests.
The host test checks that a request larger than the static scratch is
refused before anything is launched. This file is named to be collected last.
"""

import ctypes

import pytest
import torch

from _parity import assert_loss, gpu_or_skip
from vocab_ce_gb300 import workloads as wl
from vocab_ce_gb300._lib import lib

P = ctypes.c_void_p


def _call_static(H, E, y, v_valid, t, loss, lse):
    T, h = H.shape
    st = lib().vocab_parallel_ce_loss_static(P(H.data_ptr()), P(E.data_ptr()), P(y.data_ptr()), T, h, E.shape[0],
                                             v_valid, t, 0, P(loss.data_ptr()),
                                             None if lse is None else P(lse.data_ptr()),
                                             P(torch.cuda.current_stream().cuda_stream))
    return st


@pytest.mark.gpu
def test_static_scratch_forward_matches_workspace_forward_twice():
    dev = gpu_or_skip()
    import vocab_ce_gb300 as tp

    cases = [
        # (T, h, v_pad, v_valid, t): 256-wide tiles, then 128-wide tiles with lse kept internal
        (1000, 256, 4096, 3900, 8),
        (333, 200, 768, 700, 2),
    ]
    for i, (T, h, v_pad, v_valid, t) in enumerate(cases):
        w = wl.custom(f"static{i}", T=T, h=h, f=0, v_valid=v_valid, v_pad=v_pad, t=t)
        ci = {k: v.to(dev) for k, v in wl.ce_inputs(w, seed=10 + i).items()}
        ref = tp.vocab_parallel_ce(ci["H"], ci["E"], ci["targets"], v_valid, t, grads=False)
        loss = torch.full((T,), float("nan"), dtype=torch.float32, device=dev)
        lse = torch.full((T,), float("nan"), dtype=torch.float32, device=dev) if i == 0 else None
        st = _call_static(ci["H"], ci["E"], ci["targets"], v_valid, t, loss, lse)
        assert st == 0, lib().tpce_last_error()
        torch.cuda.synchronize()
        assert tp.device_status() == 0
        assert_loss("static loss", loss, ref["loss"])
        if lse is not None:
            assert_loss("static lse", lse, ref["lse"])


def test_static_scratch_refuses_oversize_request_before_launch():
    # 16,384 tokens x 504 vocabulary tiles need 66 MB of statistics: refused on
    # the host (pointers are never dereferenced on this path)
    fake = P(1 << 20)
    st = lib().vocab_parallel_ce_loss_static(fake, fake, fake, 16384, 8192, 129024, 128256, 8, 0, fake, fake, None)
    assert st == 4  # TPCE_ERR_WORKSPACE
    msg = lib().tpce_last_error().decode()
    assert "static scratch" in msg and str(16 << 20) in msg
