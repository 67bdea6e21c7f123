"""vocab_parallel_ce_loss_static: the fused cross-entropy forward for callers
that cannot allocate device memory -- a plugin whose host framework's memory
planner owns every device buffer and forbids allocations it did not plan, or
a latency-critical path that must not risk the implicit synchronisation of a
cudaMalloc. It takes no workspace: its scratch is a static device array
inside the library, shared by every call.

The GPU tests call it through the C ABI into caller-owned buffers allocated
before the calls and compare each result with vocab_parallel_ce (the
workspace version) on the same inputs, within the loss tolerance of the
parity tests:

* two calls in a row on the same shapes, the second with other targets, so
  that nothing the first call left in the shared array leaks into the second;
* then a smaller call (fewer tokens, another shard count, lse kept internal)
  after the larger ones;
* the device's free memory (cudaMemGetInfo) is the same before and after a
  call, once the first call has committed the array;
* an fp32 (tf32) case, and one call through the Python wrapper;
* one case is also checked against the CPU oracle;
* the 129K-vocabulary config (16,384 tokens) fits the array and matches.

The host test checks that a request larger than the static scratch is
refused before anything is launched. This file is named to be collected last.
"""

import ctypes

import pytest
import torch

import oracle
from _parity import assert_loss, gpu_or_skip
from vocab_ce_gb300 import workloads as wl
from vocab_ce_gb300._lib import lib

P = ctypes.c_void_p
TPCE_F32 = 1


def _call_static(H, E, y, v_valid, t, loss, lse):
    T, h = H.shape
    dt = TPCE_F32 if H.dtype == torch.float32 else 0
    return lib().vocab_parallel_ce_loss_static(P(H.data_ptr()), P(E.data_ptr()), P(y.data_ptr()), T, h, E.shape[0],
                                               v_valid, t, dt, P(loss.data_ptr()),
                                               None if lse is None else P(lse.data_ptr()),
                                               P(torch.cuda.current_stream().cuda_stream))


def _inputs(dev, T, h, v_pad, v_valid, t, seed, dtype="bf16"):
    w = wl.custom(f"static{seed}", T=T, h=h, f=0, v_valid=v_valid, v_pad=v_pad, t=t, dtype=dtype)
    return w, {k: v.to(dev) for k, v in wl.ce_inputs(w, seed=seed).items()}


def _check(tp, name, ci, v_valid, t, loss, lse):
    ref = tp.vocab_parallel_ce(ci["H"], ci["E"], ci["targets"], v_valid, t, grads=False)
    assert_loss(f"{name} loss", loss, ref["loss"])
    if lse is not None:
        assert_loss(f"{name} lse", lse, ref["lse"])


@pytest.mark.gpu
def test_static_scratch_forward_matches_workspace_forward():
    dev = gpu_or_skip()
    import vocab_ce_gb300 as tp

    # 256-wide vocabulary tiles (v_pad / t = 512), lse returned
    T, h, v_pad, v_valid, t = 1000, 256, 4096, 3900, 8
    w, ci = _inputs(dev, T, h, v_pad, v_valid, t, seed=10)
    loss = torch.full((T,), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((T,), float("nan"), dtype=torch.float32, device=dev)

    # first call: commits the static array on this device
    assert _call_static(ci["H"], ci["E"], ci["targets"], v_valid, t, loss, lse) == 0, lib().tpce_last_error()
    torch.cuda.synchronize()
    assert tp.device_status() == 0
    _check(tp, "static call 1", ci, v_valid, t, loss, lse)

    # second call, same shapes, other targets: nothing allocated, nothing left over from call 1
    g = torch.Generator().manual_seed(99)
    ci["targets"] = torch.randint(0, v_valid, (T,), generator=g, dtype=torch.int32).to(dev)
    loss.fill_(float("nan"))
    lse.fill_(float("nan"))
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    assert _call_static(ci["H"], ci["E"], ci["targets"], v_valid, t, loss, lse) == 0, lib().tpce_last_error()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert tp.device_status() == 0
    _check(tp, "static call 2 (other targets)", ci, v_valid, t, loss, lse)

    # the same inputs against the CPU oracle
    o = oracle.ce(ci["H"].cpu(), ci["E"].cpu(), ci["targets"].cpu().numpy(), v_valid, grads=False)
    assert_loss("static call 2 vs oracle", loss, o["loss"])

    # a smaller call after the larger ones: 128-wide tiles (v_pad / t = 384), lse kept internal
    T2, h2, v_pad2, v_valid2, t2 = 333, 200, 768, 700, 2
    _, c2 = _inputs(dev, T2, h2, v_pad2, v_valid2, t2, seed=11)
    loss2 = torch.full((T2,), float("nan"), dtype=torch.float32, device=dev)
    assert _call_static(c2["H"], c2["E"], c2["targets"], v_valid2, t2, loss2, None) == 0, lib().tpce_last_error()
    torch.cuda.synchronize()
    assert tp.device_status() == 0
    _check(tp, "static smaller call", c2, v_valid2, t2, loss2, None)


@pytest.mark.gpu
def test_static_scratch_fp32_and_python_wrapper():
    dev = gpu_or_skip()
    import vocab_ce_gb300 as tp

    # fp32 inputs run on the tf32 tensor path
    T, h, v_pad, v_valid, t = 96, 64, 512, 500, 2
    _, ci = _inputs(dev, T, h, v_pad, v_valid, t, seed=12, dtype="f32")
    loss = torch.full((T,), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((T,), float("nan"), dtype=torch.float32, device=dev)
    assert _call_static(ci["H"], ci["E"], ci["targets"], v_valid, t, loss, lse) == 0, lib().tpce_last_error()
    torch.cuda.synchronize()
    assert tp.device_status() == 0
    _check(tp, "static fp32", ci, v_valid, t, loss, lse)

    # the Python wrapper marshals the same call (bf16, caller-owned outputs)
    T, h, v_pad, v_valid, t = 640, 128, 2048, 2000, 4
    _, cb = _inputs(dev, T, h, v_pad, v_valid, t, seed=13)
    loss = torch.empty(T, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    res = tp.vocab_parallel_ce_loss_static(cb["H"], cb["E"], cb["targets"], v_valid, t, loss, lse)
    torch.cuda.synchronize()
    assert tp.device_status() == 0
    assert res["loss"] is loss and res["lse"] is lse
    _check(tp, "static via the Python wrapper", cb, v_valid, t, loss, lse)


@pytest.mark.gpu
def test_static_scratch_serves_the_129k_vocabulary_config():
    # 16,384 tokens over 129,024 padded ids (t = 8): 72 statistics parts per
    # token, 9.6 MB of the 16 MiB array
    dev = gpu_or_skip()
    import vocab_ce_gb300 as tp

    w = wl.WORKLOADS["ce128k"]
    ci = wl.ce_inputs(w, seed=0, device=dev)
    loss = torch.full((w.T,), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((w.T,), float("nan"), dtype=torch.float32, device=dev)
    assert _call_static(ci["H"], ci["E"], ci["targets"], w.v_valid, w.t, loss, lse) == 0, lib().tpce_last_error()
    torch.cuda.synchronize()
    assert tp.device_status() == 0
    _check(tp, "static at the 129K config", ci, w.v_valid, w.t, loss, lse)


def test_static_scratch_refuses_oversize_request_before_launch():
    # 300,000 tokens over 129,024 ids: one part per shard already needs
    # 8 x 300,000 x 8 bytes = 19.2 MB of statistics: refused on the host
    # (pointers are never dereferenced on this path)
    fake = P(1 << 20)
    st = lib().vocab_parallel_ce_loss_static(fake, fake, fake, 300000, 8192, 129024, 128256, 8, 0, fake, fake, None)
    assert st == 4  # TPCE_ERR_WORKSPACE
    msg = lib().tpce_last_error().decode()
    assert "static scratch" in msg and str(16 << 20) in msg
