"""Shared comparison helpers for the GPU parity tests.

Tolerances (fp32 accumulation, bf16 storage):
  * GEMM outputs and gradients: per tensor, max|gpu - oracle| / max|oracle| <= 1e-2.
  * Per-token loss (and lse): max|gpu - oracle| <= 2e-3 absolute.
"""

import numpy as np
import torch

REL_TOL = 1e-2
LOSS_ABS_TOL = 2e-3


def as_f64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def rel_err(gpu, ref) -> float:
    g, r = as_f64(gpu), as_f64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    denom = np.abs(r).max()
    return float(np.abs(g - r).max() / max(denom, 1e-30))


def assert_rel(name, gpu, ref, tol=REL_TOL):
    e = rel_err(gpu, ref)
    assert e <= tol, f"{name}: max rel err {e:.3e} > {tol}"
    return e


def assert_loss(name, gpu, ref, tol=LOSS_ABS_TOL):
    g, r = as_f64(gpu), as_f64(ref)
    assert np.all(np.isfinite(g)), f"{name}: non-finite"
    e = float(np.abs(g - r).max())
    assert e <= tol, f"{name}: max abs err {e:.3e} > {tol}"
    return e


def gpu_or_skip():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
