"""A bounded device wait that runs out, and the context after it.

Every wait inside the library's kernels has a time bound. The pages'
"Megatron-LM, in depth" page ("Failure modes") treats a stalled exchange as
a failure to detect, not to wait out; here the exchange is on-chip, and the
only way a kernel can stall is a barrier whose arrival never comes. This
test makes that happen on purpose, without any fault: the failure-path knob
tpce_debug_withhold_next_load(1) makes the next CTA-pair GEMM arm the full
barrier of its first k-block and load nothing into it, so the MMA thread's
wait can never complete. The test checks that

* the call returns, after the wait bound (2 s) and well before any outer limit;
* the device status word reads TPCE_ERR_TIMEOUT, naming one of the waits that
  depend on the withheld stage (the MMA thread's wait on it, or the partner
  CTA's epilogue wait on the accumulator the MMA never commits);
* the context is still usable: the same call again is clean (status 0) and
  matches the oracle, and the knob was used up by the one launch.

The case is one 256 x 256 output tile with two k-blocks (K = 128), so the
whole launch is one cluster whose pipeline never needs a stage back: no
producer waits on the stalled MMA thread, and every load it issued has landed
long before the bound runs out.
"""

import time

import pytest
import torch

import oracle
import vocab_ce_gb300 as tp
from _parity import assert_rel, gpu_or_skip
from vocab_ce_gb300 import workloads as wl
from vocab_ce_gb300._lib import lib

pytestmark = pytest.mark.gpu

TPCE_ERR_TIMEOUT = 6
WAIT_MMA_FULL = 3     # the MMA thread's wait for a loaded stage
WAIT_EPI_TFULL = 4    # an epilogue warp's wait for a finished accumulator


def _case(dev):
    w = wl.custom("timeout", T=256, h=128, f=0, v_valid=0, v_pad=0, t=2)
    g = torch.Generator().manual_seed(77)
    X = torch.randn(w.T, 128, generator=g).to(torch.bfloat16)
    W = (0.05 * torch.randn(128, 256, generator=g)).to(torch.bfloat16)
    b = (0.1 * torch.randn(256, generator=g)).float()
    return X, W, b, (X.to(dev), W.to(dev), b.to(dev))


def test_withheld_stage_times_out_and_the_context_stays_usable():
    dev = gpu_or_skip()
    X, W, b, (Xd, Wd, bd) = _case(dev)
    assert tp.device_status(clear=True) == 0  # start from a clean word
    ref = oracle.linear_forward(X, W, b)

    assert lib().tpce_debug_withhold_next_load(1) == 0
    t0 = time.perf_counter()
    tp.tp_linear_forward(Xd, Wd, 2, "column", bd)
    code, detail = tp.device_status_detail(clear=True)  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert code == TPCE_ERR_TIMEOUT, (code, hex(detail))
    assert (detail >> 8) & 0xff in (WAIT_MMA_FULL, WAIT_EPI_TFULL), hex(detail)
    assert 1.5 < elapsed < 60.0, elapsed

    # the same call again: no fault left behind, the knob is spent, the result is right
    for rep in range(2):
        Y = tp.tp_linear_forward(Xd, Wd, 2, "column", bd)
        assert tp.device_status(clear=True) == 0
        assert_rel(f"Y after a timed-out launch, call {rep}", Y, ref)


def test_disarmed_knob_changes_nothing():
    dev = gpu_or_skip()
    X, W, b, (Xd, Wd, bd) = _case(dev)
    assert lib().tpce_debug_withhold_next_load(1) == 0
    assert lib().tpce_debug_withhold_next_load(0) == 0
    Y = tp.tp_linear_forward(Xd, Wd, 2, "column", bd)
    assert tp.device_status(clear=True) == 0
    assert_rel("Y with the knob disarmed", Y, oracle.linear_forward(X, W, b))
