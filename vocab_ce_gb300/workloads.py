"""Workload table and seeded synthetic inputs.

This module holds the five workloads this library is measured and tested on
and the seeded generators that draw their inputs. It holds none of the
method's arithmetic: no GEMM, no GeLU, no softmax. Both the CUDA path (through
the tests and ``bench.py``) and the CPU oracle (through the tests) consume the
arrays made here, so that the two sides see bit-identical inputs.

Recipe (every workload):

* Activations X, H and the upstream gradient dZ are N(0, 1).
* Weights A, B, E are N(0, 0.02) -- the initialisation stated on the
  Megatron-LM digest page ("Key takeaways", initialisation bullet). B is the
  weight that feeds the residual, so it is further scaled by 1/sqrt(2N), N
  counting the attention and MLP blocks of the model the shapes come from.
* Biases are zero (a bias pin in the tests sets them non-zero explicitly).
* Targets are uniform over the real (unpadded) vocabulary ids [0, v_valid).
* bf16 workloads draw fp32 normals and round them to bf16 (round to nearest
  even); the fp32 workload keeps the fp32 draws.

Each tensor has its own generator, seeded with ``seed * 16 + slot`` where the
slot is fixed per tensor name, so drawing one tensor never shifts another.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

# fixed generator slot per tensor
_SLOTS = {"X": 1, "A": 2, "B": 3, "dZ": 4, "H": 5, "E": 6, "targets": 7, "Wqkv": 8, "Wo": 9, "O": 10,
          "dQKV": 11}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One workload: token count, widths, shard count and input statistics."""

    name: str
    T: int                 # tokens = b * s
    h: int                 # hidden width
    f: int                 # MLP inner width (0: no MLP in this workload)
    v_valid: int           # real vocabulary size (0: no CE in this workload)
    v_pad: int             # padded vocabulary (a multiple of 128 * t)
    t: int                 # tensor-parallel shards laid out on the one GPU
    dtype: str             # "bf16" or "f32"
    n_blocks: int          # attention + MLP blocks, for the 1/sqrt(2N) scaling of B
    b: int = 0
    s: int = 0
    weight_std: float = 0.02
    act: str = "gelu"      # the MLP's nonlinearity: "gelu" or "swiglu"
    chain: bool = False    # the MLP's Z is the CE's H and the CE's dH the MLP's dZ
    ce_grads: bool = True  # False: the CE is the forward-only (evaluation) loss
    sp: bool = False       # sequence-parallel entry/exit: X, Z, dZ, dX as t sequence chunks
    n_heads: int = 0       # attention projections: query heads (0: none in this workload)
    n_kv_heads: int = 0    # key/value heads (grouped-query attention)
    head_dim: int = 0

    @property
    def b_scale(self) -> float:
        return 1.0 / math.sqrt(2.0 * self.n_blocks)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


# The five workloads. Shapes follow the pages: the 8.3B GPT-2-style model of
# the Megatron-LM digest (hidden 3072, 72 layers, vocabulary 50,257 padded to
# 51,200 at 8-way), the 70B decoder of the in-depth page's worked example
# (hidden 8192, 80 layers, sequence 4096), and a 128,256-token vocabulary
# padded to a multiple of 128 * t.
WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", T=32, h=64, f=256, v_valid=512, v_pad=512, t=2,
                     dtype="f32", n_blocks=2, b=2, s=16),
    "gpt8b": Workload("gpt8b", T=8192, h=3072, f=12288, v_valid=50257, v_pad=51200,
                      t=8, dtype="bf16", n_blocks=144, b=8, s=1024),
    "mlp70b": Workload("mlp70b", T=4096, h=8192, f=32768, v_valid=0, v_pad=0, t=8,
                       dtype="bf16", n_blocks=160, b=1, s=4096),
    "ce128k": Workload("ce128k", T=16384, h=8192, f=0, v_valid=128256, v_pad=129024,
                       t=8, dtype="bf16", n_blocks=160, b=4, s=4096),
    # the SwiGLU block of the Llama-3-70B page (hidden 8192, TP 8, sequence
    # 4096); the page gives no FFN width, the model's published 28,672 is used
    "swiglu70b": Workload("swiglu70b", T=4096, h=8192, f=28672, v_valid=0, v_pad=0, t=8,
                          dtype="bf16", n_blocks=160, b=1, s=4096, act="swiglu"),
    # the attention projections of the same model: 64 query heads sharing 8
    # key/value heads of width 128 (the page's figures), t = 8
    "attn70b": Workload("attn70b", T=4096, h=8192, f=0, v_valid=0, v_pad=0, t=8, dtype="bf16",
                        n_blocks=160, b=1, s=4096, n_heads=64, n_kv_heads=8, head_dim=128),
}

# the 8.3B block chained into its head (last layer + loss, a training step),
# and the 128,256-token loss forward only (evaluation)
WORKLOADS["gpt8b_chain"] = dataclasses.replace(WORKLOADS["gpt8b"], name="gpt8b_chain", chain=True)
WORKLOADS["ce128k_eval"] = dataclasses.replace(WORKLOADS["ce128k"], name="ce128k_eval", ce_grads=False)
# the 70B MLP with sequence-parallel entry and exit (t = 8 chunks of 512 tokens)
WORKLOADS["mlp70b_sp"] = dataclasses.replace(WORKLOADS["mlp70b"], name="mlp70b_sp", sp=True)

# shard-count sweep over the 8.3B MLP shapes
SWEEP_T = (1, 2, 4, 8, 16)


def sweep_workload(t: int) -> Workload:
    base = WORKLOADS["gpt8b"]
    return dataclasses.replace(base, name=f"sweep_t{t}", t=t, v_valid=0, v_pad=0)


def custom(name: str, T: int, h: int, f: int, v_valid: int, v_pad: int, t: int,
           dtype: str = "bf16", n_blocks: int = 2, act: str = "gelu", n_heads: int = 0,
           n_kv_heads: int = 0, head_dim: int = 0) -> Workload:
    """A workload of arbitrary shape with the same input statistics."""
    return Workload(name, T=T, h=h, f=f, v_valid=v_valid, v_pad=v_pad, t=t,
                    dtype=dtype, n_blocks=n_blocks, act=act, n_heads=n_heads,
                    n_kv_heads=n_kv_heads, head_dim=head_dim)


def _gen(device, seed: int, slot: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 16 + _SLOTS[slot])
    return g


def _normal(shape, std, dtype, device, seed, slot):
    g = _gen(device, seed, slot)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def mlp_inputs(w: Workload, seed: int = 0, device="cpu") -> Dict[str, torch.Tensor]:
    """X [T,h], A [h,f], B [f,h] (dtype), bA [f], bB [h] (fp32 zeros), dZ [T,h]."""
    dt = w.torch_dtype
    return {
        "X": _normal((w.T, w.h), 1.0, dt, device, seed, "X"),
        "A": _normal((w.h, w.f), w.weight_std, dt, device, seed, "A"),
        "B": _normal((w.f, w.h), w.weight_std * w.b_scale, dt, device, seed, "B"),
        "bA": torch.zeros(w.f, dtype=torch.float32, device=device),
        "bB": torch.zeros(w.h, dtype=torch.float32, device=device),
        "dZ": _normal((w.T, w.h), 1.0, dt, device, seed, "dZ"),
    }


def swiglu_inputs(w: Workload, seed: int = 0, device="cpu") -> Dict[str, torch.Tensor]:
    """X [T,h], W1 = [W_gate | W_up] [h,2f], W2 [f,h] (dtype), b1 [2f], b2 [h]
    (fp32 zeros), dZ [T,h]. W1 and W2 take the generator slots of A and B."""
    dt = w.torch_dtype
    return {
        "X": _normal((w.T, w.h), 1.0, dt, device, seed, "X"),
        "W1": _normal((w.h, 2 * w.f), w.weight_std, dt, device, seed, "A"),
        "W2": _normal((w.f, w.h), w.weight_std * w.b_scale, dt, device, seed, "B"),
        "b1": torch.zeros(2 * w.f, dtype=torch.float32, device=device),
        "b2": torch.zeros(w.h, dtype=torch.float32, device=device),
        "dZ": _normal((w.T, w.h), 1.0, dt, device, seed, "dZ"),
    }


def attn_inputs(w: Workload, seed: int = 0, device="cpu") -> Dict[str, torch.Tensor]:
    """Inputs of the attention projections: X [T,h], Wqkv [h,(n_q+2 n_kv) d],
    O [T, n_q d] (the attention core's output, which this library does not
    compute, drawn N(0,1)), Wo [n_q d, h] (scaled like B: it feeds the
    residual), upstream gradients dQKV [T,(n_q+2 n_kv) d] and dZ [T,h], and
    zero fp32 biases bqkv, bo."""
    dt = w.torch_dtype
    nqkv = (w.n_heads + 2 * w.n_kv_heads) * w.head_dim
    hq = w.n_heads * w.head_dim
    return {
        "X": _normal((w.T, w.h), 1.0, dt, device, seed, "X"),
        "Wqkv": _normal((w.h, nqkv), w.weight_std, dt, device, seed, "Wqkv"),
        "bqkv": torch.zeros(nqkv, dtype=torch.float32, device=device),
        "O": _normal((w.T, hq), 1.0, dt, device, seed, "O"),
        "Wo": _normal((hq, w.h), w.weight_std * w.b_scale, dt, device, seed, "Wo"),
        "bo": torch.zeros(w.h, dtype=torch.float32, device=device),
        "dQKV": _normal((w.T, nqkv), 1.0, dt, device, seed, "dQKV"),
        "dZ": _normal((w.T, w.h), 1.0, dt, device, seed, "dZ"),
    }


def ce_inputs(w: Workload, seed: int = 0, device="cpu") -> Dict[str, torch.Tensor]:
    """H [T,h], E [v_pad,h] (dtype), targets [T] int32 uniform over [0, v_valid)."""
    dt = w.torch_dtype
    g = _gen(device, seed, "targets")
    targets = torch.randint(0, w.v_valid, (w.T,), generator=g, device=device,
                            dtype=torch.int64).to(torch.int32)
    return {
        "H": _normal((w.T, w.h), 1.0, dt, device, seed, "H"),
        "E": _normal((w.v_pad, w.h), w.weight_std, dt, device, seed, "E"),
        "targets": targets,
    }


def sample_indices(n: int, k: int, seed: int = 0, include_edges: bool = True) -> torch.Tensor:
    """k distinct indices in [0, n), sorted; the first and last index included."""
    k = min(k, n)
    g = torch.Generator().manual_seed(seed + 12345)
    idx = torch.randperm(n, generator=g)[:k]
    if include_edges and k >= 2:
        idx[0] = 0
        idx[1] = n - 1
        idx = torch.unique(idx)
    return torch.sort(idx).values


def to_f32_numpy(x: torch.Tensor):
    """Exact widening of bf16/fp32 data to a contiguous fp32 numpy array."""
    return x.detach().to("cpu").to(torch.float32).contiguous().numpy()


def maybe_int32_numpy(x: Optional[torch.Tensor]):
    return None if x is None else x.detach().to("cpu").to(torch.int32).contiguous().numpy()
