#!/usr/bin/env python
"""Benchmark: tensor-parallel MLP block forward+backward and fused
vocabulary-parallel cross-entropy forward+backward, all t shards on one GPU.

One step = one pass of the whole path over one batch of synthetic inputs
resident in HBM. The default workload, ``headline``, is the pair of
configurations the targets are stated on, run back to back in every step:

* the 70B-shaped GeLU MLP block forward+backward (T = 4096 tokens, h = 8192,
  f = 32768, t = 8): tp_mlp_forward, tp_mlp_backward;
* the fused vocabulary-parallel logit GEMM + cross-entropy forward+backward
  over a 128,256-id vocabulary padded to 129,024 (T = 16,384, h = 8192,
  t = 8): vocab_parallel_ce with loss, dH and dE.

Printed (rank 0, one JSON line): whole-job TFLOP/s over the step (MLP
12 T h f + CE 8 T h v_pad FLOPs, the CE count including the logit recompute
that unmaterialised logits require), the MLP TFLOP/s and CE tokens/s parts
with their fractions of the dense bf16 peak (2.25 PFLOP/s nominal, and the
measured burst and sustained figures), the end-to-end figure through the
Python API from pinned host buffers, the roofline of the dominant kernel,
SM clocks during the timed region, and the CPU oracle timed on a bounded
sample on this host.

The headline timing runs with the library's kernel timer off; the per-kernel
figures (and the dominant kernel's roofline) come from a second pass of the
same steps with the timer on, right after.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W]
                       [--impl ours|reference]
                       [--workload headline|gpt8b|gpt8b_chain|mlp70b|mlp70b_sp|ce128k|ce128k_eval|
                                   swiglu70b|attn70b|sweep]
Multi-GPU (one process per GPU under torchrun): every rank runs its own
independent batch (data parallel, weak scaling); there is no collective on
the data path, only a barrier and a max over ranks of the elapsed time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from vocab_ce_gb300 import workloads as wl  # noqa: E402

METRIC = "TP-MLP fwd+bwd TFLOP/s and fused vocab-parallel CE tokens/s vs roofline, 1 GB300"
UNIT = "TFLOP/s"
# fallbacks only if the generated MEASURED_PEAKS.json is absent
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal dense bf16 tensor peak of a GB300, the figure the targets are stated against
SPEC_BF16_TFLOPS = 2250.0
# targets: MLP at >= 60% of the dense bf16 peak, fused CE at >= 50% of its roofline
TARGETS = {"mlp_frac_of_spec_peak": 0.60, "ce_frac_of_spec_roofline": 0.50}
# a timed region at least this long runs under the power cap: its kernels are
# compared with the measured sustained peak, shorter ones with the burst peak
SUSTAINED_REGION_S = 1.0

# the pages' own figures, quoted beside the line as context (other hardware, whole-model
# training on clusters; none is a figure for this path on one GPU)
PAGES_CONTEXT = ("8.3B-parameter GPT-2-style model, 8-way tensor parallel x data parallel on 512 GPUs: 15.1 PFLOP/s "
                 "aggregate, 76% scaling efficiency against a 39 TFLOP/s single-GPU baseline; 1T-parameter model with "
                 "tensor + pipeline + data parallelism on 3,072 A100s: 502 PFLOP/s (52% of peak)")

# the workloads of each job, run back to back in one step
JOBS = {"headline": ("mlp70b", "ce128k")}
WORKLOAD_NAMES = ["headline", "gpt8b", "gpt8b_chain", "mlp70b", "mlp70b_sp", "ce128k", "ce128k_eval", "swiglu70b",
                  "attn70b", "sweep"]
# tokens of each workload the CPU oracle processes per timed sample
CPU_SAMPLE_TOKENS = {"gpt8b": 512, "gpt8b_chain": 512, "mlp70b": 192, "mlp70b_sp": 192, "ce128k": 96, "ce128k_eval": 256,
                     "swiglu70b": 144, "attn70b": 512, "sweep": 512}
CPU_SAMPLE_TOKENS_JOB = {"headline": {"mlp70b": 96, "ce128k": 48}}
REF_STEP_TOKENS = {"gpt8b": 8, "gpt8b_chain": 8, "mlp70b": 4, "mlp70b_sp": 4, "ce128k": 2, "ce128k_eval": 4, "swiglu70b": 3,
                   "attn70b": 8, "sweep": 8}
REF_STEP_TOKENS_JOB = {"headline": {"mlp70b": 1, "ce128k": 2}}


# ---------------------------------------------------------------------- setup
def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=WORKLOAD_NAMES, default="headline")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--no-kernel-pass", action="store_true", help="skip the per-kernel timing pass")
    p.add_argument("--tokens", type=int, default=0,
                   help="run every workload of the job on this many tokens instead of its own T (a smaller "
                        "case of the same kernels, for profiler captures); the line then names the reduced T")
    return p.parse_args(argv)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device) -> float:
    """The largest of every rank's value (each rank's elapsed time -> the job's)."""
    if ws <= 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(ws: int, work_per_rank: float, seconds: float) -> float:
    """Whole-job throughput: the work all ranks processed over the slowest rank's time."""
    return ws * work_per_rank / seconds


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def job_workloads(name, tokens=0):
    """The workloads one step of job `name` runs, in launch order (on `tokens`
    tokens each when given, else at their own T)."""
    import dataclasses

    ws_ = [wl.WORKLOADS[n] for n in JOBS.get(name, (name,))]
    return [dataclasses.replace(w, T=tokens, b=1, s=tokens) for w in ws_] if tokens else ws_


def flops(w):
    """(MLP-side, CE-side) FLOPs of one step of workload w, in the bench's convention."""
    # GeLU block: 4 T h f forward + 8 T h f backward; SwiGLU: GEMM1 is twice as
    # wide (6 T h f forward, 12 T h f backward)
    mlp = (18.0 if w.act == "swiglu" else 12.0) * w.T * w.h * w.f if w.f else 0.0
    # CE: 2 T h v_pad for the logits, 6 more with gradients (recompute, dE, dH)
    ce = (8.0 if w.ce_grads else 2.0) * w.T * w.h * w.v_pad if w.v_pad else 0.0
    # attention projections: QKV and W_O, each forward + dX + dW
    if w.n_heads:
        nqkv = (w.n_heads + 2 * w.n_kv_heads) * w.head_dim
        mlp += 6.0 * w.T * w.h * nqkv + 6.0 * w.T * (w.n_heads * w.head_dim) * w.h
    return mlp, ce


def ce_model_flops(w):
    """CE model FLOPs over the real vocabulary without the backward's logit
    recompute: 6 T h v_valid with gradients (logits, dH, dE), 2 T h v_valid
    for the loss alone."""
    return ((6.0 if w.ce_grads else 2.0) * w.T * w.h * w.v_valid) if w.v_pad else 0.0


def job_flops(ws_):
    mlp = sum(flops(w)[0] for w in ws_)
    ce = sum(flops(w)[1] for w in ws_)
    return mlp, ce


def workload_config(w, name):
    desc = {
        "gpt8b": "8.3B-shaped block: MLP fwd+bwd + fused vocab-parallel CE fwd+bwd",
        "gpt8b_chain": "8.3B-shaped block chained into its loss: MLP fwd, CE fwd+bwd on H = Z, MLP bwd with dZ = dH",
        "ce128k_eval": "vocab-parallel fused logit GEMM + CE forward only (per-token loss), 128,256-token vocabulary",
        "mlp70b": "70B-shaped MLP fwd+bwd",
        "mlp70b_sp": "70B-shaped MLP fwd+bwd with sequence-parallel entry/exit (X, Z, dZ, dX as t sequence chunks)",
        "ce128k": "vocab-parallel fused logit GEMM + CE fwd+bwd, 128,256-token vocabulary",
        "swiglu70b": "70B-shaped SwiGLU MLP fwd+bwd (gate/up column-parallel, down row-parallel)",
        "attn70b": "70B-shaped attention projections fwd+bwd (QKV column-parallel by GQA heads, W_O row-parallel; "
                   "attention core excluded)",
        "sweep": "shard-count sweep of the 8.3B MLP fwd+bwd",
    }[name]
    cfg = {"workload": f"{desc}: T={w.T} (b={w.b}, s={w.s}), h={w.h}", "T": w.T, "h": w.h, "t": w.t,
           "seed": 0, "inputs": "seeded synthetic (workloads.py recipe), resident in HBM"}
    if w.f:
        cfg["f"] = w.f
    if w.v_pad:
        cfg.update(v_valid=w.v_valid, v_pad=w.v_pad)
    if w.n_heads:
        cfg.update(n_heads=w.n_heads, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim)
    return cfg


def job_config(name, ws_):
    """The `config` of a job: one workload's, or for a composite job a
    description naming every part and each part's own config."""
    if len(ws_) == 1:
        return workload_config(ws_[0], name)
    parts = {w.name: workload_config(w, w.name) for w in ws_}
    m, c = ws_
    text = (f"70B-shaped MLP fwd+bwd (T={m.T}, h={m.h}, f={m.f}, GeLU, t={m.t}) then vocab-parallel fused logit GEMM "
            f"+ CE fwd+bwd (T={c.T}, h={c.h}, vocabulary {c.v_valid:,} padded to {c.v_pad:,}, t={c.t}), each step")
    return {"workload": text, "parts": parts, "seed": 0,
            "inputs": "seeded synthetic (workloads.py recipe), resident in HBM"}


# ---------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device, enabled=True):
        self.proc = None
        self.path = None
        if not enabled:
            return
        sel = []
        try:
            uuid = torch.cuda.get_device_properties(device).uuid
            sel = ["-i", "GPU-" + str(uuid)]
        except Exception:
            pass
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50"] + sel, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                power = float(parts[3])
            except ValueError:
                power = None
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9], power))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r, _ in rows for i in range(4) if r[i].lower().startswith("active")})
        watts = [r[3] for r in rows if r[3] is not None]
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows),
                "power_w_median": statistics.median(watts) if watts else None}


# ---------------------------------------------------------------------- traffic from committed ncu summaries
# The translation unit each kernel's launch is compiled in (by name prefix).
KERNEL_UNITS = (("ce_static_", "ce_static.cu"), ("ce_", "ce.cu"), ("mlp_", "mlp.cu"), ("swiglu_", "mlp.cu"),
                ("linear_", "linear.cu"), ("attn_", "linear.cu"), ("transpose_", "runtime.cu"),
                ("colsum_", "runtime.cu"), ("f32_to_bf16", "runtime.cu"))


def _code_only(text):
    """A CUDA source without its comments and with whitespace runs collapsed:
    what the compiler sees, so that editing a comment keeps the hash."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel=None):
    """A hash over the code a kernel is built from: its translation unit and
    every shared header of the library (every CUDA source when the kernel is
    not known), comments left out. Recorded traffic is only trusted for the
    code it was captured with."""
    d = os.path.join(ROOT, "vocab_ce_gb300", "csrc")
    unit = next((u for p, u in KERNEL_UNITS if kernel and kernel.startswith(p)), None)
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        if f.endswith((".cuh", ".h")) or (f.endswith(".cu") and unit in (None, f)):
            with open(os.path.join(d, f), encoding="utf-8") as fh:
                h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel, workload):
    """dram bytes per launch recorded in profiles/ for this kernel and workload,
    if the kernel's sources have not changed since the capture; else None."""
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    src = kernel_source_hash(kernel)
    for fn in sorted(os.listdir(d)):
        if not fn.endswith((".md", ".txt")):
            continue
        text = open(os.path.join(d, fn)).read()
        for m in re.finditer(r"traffic_per_launch\s+kernel=(\S+)\s+workload=(\S+)\s+bytes=(\d+)\s+source=(\w+)",
                             text):
            if m.group(1) == kernel and m.group(2) == workload and m.group(4) == src:
                return int(m.group(3))
    return None


# ---------------------------------------------------------------------- the step
class Step:
    def __init__(self, w, dev, seed):
        import vocab_ce_gb300 as tp

        self.tp = tp
        self.w = w
        self.dev = dev
        self.glu = w.act == "swiglu"
        if not w.f:
            self.mi = None
        else:
            self.mi = (wl.swiglu_inputs if self.glu else wl.mlp_inputs)(w, seed=seed, device=dev)
        if w.f and w.sp:
            # one buffer per rank's sequence chunk of X and dZ
            rows = w.T // w.t
            for k in ("X", "dZ"):
                full = self.mi.pop(k)
                for r in range(w.t):
                    self.mi[f"{k}{r}"] = full[r * rows:(r + 1) * rows].clone()
        self.ci = wl.ce_inputs(w, seed=seed, device=dev) if w.v_pad else None
        self.ai = wl.attn_inputs(w, seed=seed, device=dev) if w.n_heads else None
        T, h, f = w.T, w.h, w.f
        bf = torch.bfloat16
        self.out = {}
        if w.f and not self.glu:
            self.fo = {k: torch.empty(s, dtype=bf, device=dev) for k, s in (("Z", (T, h)), ("U", (T, f)), ("Y", (T, f)))}
            if w.sp:
                rows = T // w.t
                self.zc = [torch.empty((rows, h), dtype=bf, device=dev) for _ in range(w.t)]
                self.dxc = [torch.empty((rows, h), dtype=bf, device=dev) for _ in range(w.t)]
            self.bo = {"dX": torch.empty((T, h), dtype=bf, device=dev), "dA": torch.empty((h, f), dtype=bf, device=dev),
                       "dB": torch.empty((f, h), dtype=bf, device=dev),
                       "dbA": torch.empty(f, dtype=torch.float32, device=dev),
                       "dbB": torch.empty(h, dtype=torch.float32, device=dev)}
            self.mws = torch.empty(max(1, tp.mlp_workspace_bytes(T, h, f, w.t)), dtype=torch.uint8, device=dev)
        elif w.f:
            self.fo = {k: torch.empty(s, dtype=bf, device=dev)
                       for k, s in (("Z", (T, h)), ("GU", (T, 2 * f)), ("Y", (T, f)))}
            self.bo = {"dX": torch.empty((T, h), dtype=bf, device=dev),
                       "dW1": torch.empty((h, 2 * f), dtype=bf, device=dev),
                       "dW2": torch.empty((f, h), dtype=bf, device=dev),
                       "db1": torch.empty(2 * f, dtype=torch.float32, device=dev),
                       "db2": torch.empty(h, dtype=torch.float32, device=dev)}
            self.mws = torch.empty(max(1, tp.swiglu_workspace_bytes(T, h, f, w.t)), dtype=torch.uint8, device=dev)
        if w.n_heads:
            nqkv = (w.n_heads + 2 * w.n_kv_heads) * w.head_dim
            hq = w.n_heads * w.head_dim
            self.ao = {"QKV": torch.empty((T, nqkv), dtype=bf, device=dev), "Z": torch.empty((T, h), dtype=bf, device=dev)}
            self.aq = {"dX": torch.empty((T, h), dtype=bf, device=dev), "dWqkv": torch.empty((h, nqkv), dtype=bf, device=dev),
                       "dbqkv": torch.empty(nqkv, dtype=torch.float32, device=dev)}
            self.ag = {"dO": torch.empty((T, hq), dtype=bf, device=dev), "dWo": torch.empty((hq, h), dtype=bf, device=dev),
                       "dbo": torch.empty(h, dtype=torch.float32, device=dev)}
            self.aws = torch.empty(max(1, tp.attn_workspace_bytes(T, h, w.n_heads, w.n_kv_heads, w.head_dim, w.t)),
                                   dtype=torch.uint8, device=dev)
        if w.v_pad:
            self.co = {"loss": torch.empty(T, dtype=torch.float32, device=dev),
                       "lse": torch.empty(T, dtype=torch.float32, device=dev)}
            if w.ce_grads:
                self.co.update(dH=torch.empty((T, h), dtype=bf, device=dev),
                               dE=torch.empty((w.v_pad, h), dtype=bf, device=dev))
            self.cws = torch.empty(tp.ce_workspace_bytes(T, h, w.v_pad, w.t, grads=w.ce_grads), dtype=torch.uint8,
                                   device=dev)
        # inputs a chained step does not read: dZ comes from the CE, H from the MLP
        self.unused = {("m", "dZ"), ("c", "H")} if w.chain else set()

    def mlp_fwd(self, mi=None):
        mi = mi or self.mi
        tp, w = self.tp, self.w
        if w.sp:
            xc = [mi[f"X{r}"] for r in range(w.t)]
            return tp.tp_mlp_forward_sp(xc, mi["A"], mi["B"], w.t, mi["bA"], mi["bB"],
                                        out={"Z": self.zc, "U": self.fo["U"], "Y": self.fo["Y"]}, ws=self.mws)
        if self.glu:
            return tp.tp_swiglu_forward(mi["X"], mi["W1"], mi["W2"], w.t, mi["b1"], mi["b2"], out=self.fo, ws=self.mws)
        return tp.tp_mlp_forward(mi["X"], mi["A"], mi["B"], w.t, mi["bA"], mi["bB"], out=self.fo, ws=self.mws)

    def mlp_bwd(self, mi=None, dZ=None):
        mi = mi or self.mi
        tp, w, fo = self.tp, self.w, self.fo
        if w.sp:
            xc = [mi[f"X{r}"] for r in range(w.t)]
            dzc = [mi[f"dZ{r}"] for r in range(w.t)]
            tp.tp_mlp_backward_sp(dzc, xc, mi["A"], mi["B"], fo["U"], fo["Y"], w.t, out={**self.bo, "dX": self.dxc},
                                  ws=self.mws)
            return
        dZ = mi["dZ"] if dZ is None else dZ
        if self.glu:
            tp.tp_swiglu_backward(dZ, mi["X"], mi["W1"], mi["W2"], fo["GU"], fo["Y"], w.t, out=self.bo, ws=self.mws)
        else:
            tp.tp_mlp_backward(dZ, mi["X"], mi["A"], mi["B"], fo["U"], fo["Y"], w.t, out=self.bo, ws=self.mws)

    def mlp(self, mi=None):
        self.mlp_fwd(mi)
        self.mlp_bwd(mi)

    def attn(self, ai=None):
        ai = ai or self.ai
        tp, w = self.tp, self.w
        nq, nkv, d = w.n_heads, w.n_kv_heads, w.head_dim
        tp.tp_attn_qkv_forward(ai["X"], ai["Wqkv"], nq, nkv, d, w.t, ai["bqkv"], out=self.ao["QKV"], ws=self.aws)
        tp.tp_attn_qkv_backward(ai["dQKV"], ai["X"], ai["Wqkv"], nq, nkv, d, w.t, out=self.aq, ws=self.aws)
        tp.tp_attn_out_forward(ai["O"], ai["Wo"], nq, d, w.t, ai["bo"], out=self.ao["Z"], ws=self.aws)
        tp.tp_attn_out_backward(ai["dZ"], ai["O"], ai["Wo"], nq, d, w.t, out=self.ag, ws=self.aws)

    def ce(self, ci=None, H=None):
        ci = ci or self.ci
        H = ci["H"] if H is None else H
        return self.tp.vocab_parallel_ce(H, ci["E"], ci["targets"], self.w.v_valid, self.w.t, grad_scale=1.0,
                                         grads=self.w.ce_grads, out=self.co, ws=self.cws)

    def segments(self, mi=None, ci=None, ai=None):
        """The step as (part, call) pairs in launch order."""
        w = self.w
        if w.chain:
            return [("mlp", lambda: self.mlp_fwd(mi)),
                    ("ce", lambda: self.ce(ci, H=self.fo["Z"])),
                    ("mlp", lambda: self.mlp_bwd(mi, dZ=self.co["dH"]))]
        seg = []
        if w.f:
            seg.append(("mlp", lambda: self.mlp(mi)))
        if w.n_heads:
            seg.append(("mlp", lambda: self.attn(ai)))
        if w.v_pad:
            seg.append(("ce", lambda: self.ce(ci)))
        return seg

    def run(self, mi=None, ci=None, ai=None):
        for _, fn in self.segments(mi, ci, ai):
            fn()


class Job:
    """The steps of every workload of a job, run back to back."""

    def __init__(self, ws_, dev, seed):
        self.steps = [Step(w, dev, seed) for w in ws_]

    def segments(self, ins=None):
        seg = []
        for k, st in enumerate(self.steps):
            mi, ci, ai = ins[k] if ins else (None, None, None)
            seg += st.segments(mi, ci, ai)
        return seg

    def run(self, ins=None):
        for _, fn in self.segments(ins):
            fn()


def input_bytes(step):
    b = 0
    for tag, d in (("m", step.mi), ("c", step.ci), ("a", step.ai)):
        if d:
            b += sum(v.numel() * v.element_size() for k, v in d.items() if (tag, k) not in step.unused)
    return b


# ---------------------------------------------------------------------- CPU oracle
def oracle_sample(w, mi, ci, n_tokens, ai=None):
    """Host copies of the first n_tokens tokens plus the full weights, as float64."""
    import numpy as np

    def f64(x):
        return x.detach().float().cpu().numpy().astype(np.float64)

    s = {}
    if mi is not None and "W1" in mi:
        s.update(X=f64(mi["X"][:n_tokens]), dZ=f64(mi["dZ"][:n_tokens]), W1=f64(mi["W1"]), W2=f64(mi["W2"]),
                 b1=f64(mi["b1"]), b2=f64(mi["b2"]))
    elif mi is not None:
        # sequence-parallel steps hold X and dZ as chunks: the sample is the first chunk's first tokens
        X, dZ = (mi[k] if k in mi else mi[k + "0"] for k in ("X", "dZ"))
        s.update(X=f64(X[:n_tokens]), dZ=f64(dZ[:n_tokens]), A=f64(mi["A"]), B=f64(mi["B"]),
                 bA=f64(mi["bA"]), bB=f64(mi["bB"]))
    if ci is not None:
        s.update(H=f64(ci["H"][:n_tokens]), E=f64(ci["E"]),
                 y=ci["targets"][:n_tokens].cpu().numpy().astype(np.int32))
    if ai is not None:
        s["attn"] = {k: f64(v[:n_tokens]) if k in ("X", "O", "dQKV", "dZ") else f64(v) for k, v in ai.items()}
    return s


def oracle_step(w, s):
    import oracle

    if w.chain:
        # the same chain: H = Z of the block, dZ = dH of the loss
        z = oracle.mlp_forward(s["X"], s["A"], s["bA"], s["B"], s["bB"])["Z"]
        c = oracle.ce(z, s["E"], s["y"], w.v_valid, grad_scale=1.0)
        oracle.mlp_backward(s["X"], s["A"], s["bA"], s["B"], c["dH"])
        return
    if "W1" in s:
        oracle.swiglu_forward(s["X"], s["W1"], s["b1"], s["W2"], s["b2"])
        oracle.swiglu_backward(s["X"], s["W1"], s["b1"], s["W2"], s["dZ"])
    elif "X" in s:
        oracle.mlp_forward(s["X"], s["A"], s["bA"], s["B"], s["bB"])
        oracle.mlp_backward(s["X"], s["A"], s["bA"], s["B"], s["dZ"])
    if "attn" in s:
        a = s["attn"]
        oracle.linear_forward(a["X"], a["Wqkv"], a["bqkv"])
        oracle.linear_backward(a["X"], a["Wqkv"], a["dQKV"])
        oracle.linear_forward(a["O"], a["Wo"], a["bo"])
        oracle.linear_backward(a["O"], a["Wo"], a["dZ"])
    if "H" in s:
        oracle.ce(s["H"], s["E"], s["y"], w.v_valid, grad_scale=1.0, grads=w.ce_grads)


def sample_work(ws_, tokens):
    """FLOPs (bench convention) of processing tokens[w.name] tokens of each workload."""
    return sum(sum(flops(w)) / w.T * tokens[w.name] for w in ws_)


def sample_text(ws_, tokens):
    return " + ".join(f"first {tokens[w.name]} of {w.T} tokens of {w.name}" for w in ws_)


# ---------------------------------------------------------------------- arms
def run_reference(args, ws_, name):
    import oracle

    _, rank, _ = dist_env()
    if rank != 0:
        return 0
    oracle.build()
    tokens = REF_STEP_TOKENS_JOB.get(name) or {ws_[0].name: REF_STEP_TOKENS[name]}
    samples = []
    for w in ws_:
        mi = ((wl.swiglu_inputs if w.act == "swiglu" else wl.mlp_inputs)(w, seed=0)) if w.f else None
        ci = wl.ce_inputs(w, seed=0) if w.v_pad else None
        ai = wl.attn_inputs(w, seed=0) if w.n_heads else None
        samples.append((w, oracle_sample(w, mi, ci, tokens[w.name], ai)))
        del mi, ci, ai

    def step():
        for w, s in samples:
            oracle_step(w, s)

    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    dt = sum(times) / len(times)
    value = sample_work(ws_, tokens) / dt / 1e12
    sample = f"{sample_text(ws_, tokens)} per step at full h, f, v (weights in full), fp64 oracle"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": job_config(name, ws_),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def time_steps(job, steps, stream, profiled=False, clocks=None):
    """Run `steps` steps between two events on `stream`; per-segment events
    give the MLP and CE parts. Returns (elapsed ms, {part: ms per step},
    per-kernel timer records when `profiled`, else None, and the clock record
    when a sampler factory is given, else None)."""
    import vocab_ce_gb300 as tp

    segs = job.segments()
    ev = [[(part, torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for part, _ in segs]
          for _ in range(steps)]
    torch.cuda.synchronize()
    if profiled:
        tp.profile_enable(True)
    sampler = clocks() if clocks else None
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(steps):
        for (_, a, b), (_, fn) in zip(ev[i], segs):
            a.record(stream)
            fn()
            b.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = sampler.stop() if sampler else None
    kernels = None
    if profiled:
        kernels = tp.profile_read()
        tp.profile_enable(False)
    parts = {}
    for e in ev:
        for part, a, b in e:
            parts[part] = parts.get(part, 0.0) + a.elapsed_time(b)
    return t_start.elapsed_time(t_end), {k: v / steps for k, v in parts.items()}, kernels, clk


def fractions(ws_, mlp_ms, ce_ms, pk):
    """The parts of a step and their fractions of the dense bf16 peak: the
    nominal 2.25 PFLOP/s the targets are stated against, and the measured
    burst and sustained figures."""
    mlp_fl, ce_fl = job_flops(ws_)
    out = {}
    has_mlp = any(w.f for w in ws_)
    has_attn = any(w.n_heads for w in ws_)
    ce_ws = [w for w in ws_ if w.v_pad]
    denoms = {"spec": SPEC_BF16_TFLOPS, "measured_burst": pk["bf16_tflops"],
              "measured_sustained": pk["bf16_tflops_sustained"]}
    if (has_mlp or has_attn) and mlp_ms:
        r = mlp_fl / (mlp_ms * 1e-3) / 1e12
        key = "mlp" if has_mlp else "attn_proj"
        out[f"{key}_tflops"] = r
        out[f"{key}_ms"] = mlp_ms
        out[f"{key}_frac_of_spec_peak"] = r / denoms["spec"]
        out[f"{key}_frac_of_measured_burst_peak"] = r / denoms["measured_burst"]
        out[f"{key}_frac_of_measured_sustained_peak"] = r / denoms["measured_sustained"]
    if ce_ws and ce_ms:
        T = sum(w.T for w in ce_ws)
        r = ce_fl / (ce_ms * 1e-3) / 1e12
        tok = T / (ce_ms * 1e-3)
        model = sum(ce_model_flops(w) for w in ce_ws) / (ce_ms * 1e-3) / 1e12
        # the roofline in tokens/s: the peak over the FLOPs one token costs (8 h v_pad, or 2 h v_pad forward only)
        per_tok = ce_fl / T
        out.update(ce_tokens_per_s=tok, ce_ms=ce_ms, ce_tflops=r,
                   ce_roofline_tokens_per_s_spec=denoms["spec"] * 1e12 / per_tok,
                   ce_frac_of_spec_roofline=r / denoms["spec"],
                   ce_frac_of_measured_burst_roofline=r / denoms["measured_burst"],
                   ce_frac_of_measured_sustained_roofline=r / denoms["measured_sustained"],
                   ce_model_tflops=model, ce_model_frac_of_spec_peak=model / denoms["spec"],
                   ce_flop_convention=("8 T h v_pad with gradients (logits, their recompute in the backward, dE, dH; "
                                       "padded ids count, they are computed), 2 T h v_pad forward only; the model "
                                       "figure counts 6 T h v_valid (2 T h v_valid forward only): no recompute, "
                                       "real ids only"))
    return out


def run_ours(args, ws_, name):
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    import vocab_ce_gb300 as tp

    job = Job(ws_, dev, seed=rank)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        job.run()
    torch.cuda.synchronize()
    assert tp.device_status() == 0, "device status after warm-up"

    def barrier():
        if ws > 1:
            import torch.distributed as dist

            dist.barrier()

    # ---------------- timed region (device-resident inputs, kernel timer off)
    mlp_fl, ce_fl = job_flops(ws_)
    barrier()
    elapsed_ms, parts_ms, _, clk = time_steps(
        job, args.steps, stream, clocks=(lambda: ClockSampler(dev)) if not args.no_clocks else None)
    barrier()
    assert tp.device_status() == 0, "device status after the timed region"
    elapsed_ms = max_over_ranks(elapsed_ms, ws, dev)
    ms_step = elapsed_ms / args.steps
    value = job_rate(ws, mlp_fl + ce_fl, ms_step * 1e-3) / 1e12
    region_s = elapsed_ms * 1e-3

    pk, pk_src = peaks()
    sustained = region_s >= SUSTAINED_REGION_S
    peak = pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]
    peak_kind = (f"{pk_src} {'sustained' if sustained else 'burst'} bf16: the kernel runs inside a timed region of "
                 f"{region_s:.2f} s of back-to-back steps ({'>=' if sustained else '<'} {SUSTAINED_REGION_S:.0f} s)")

    # ---------------- per-kernel pass: the same steps with the library's kernel timer on
    roof, per_kernel, gpu_launches = None, None, None
    if not args.no_kernel_pass:
        barrier()
        _, _, kernels, _ = time_steps(job, args.steps, stream, profiled=True)
        barrier()
        assert tp.device_status() == 0, "device status after the kernel pass"
        dominant = max(kernels.items(), key=lambda kv: kv[1]["ms"]) if kernels else None
        if dominant:
            kname, kd = dominant
            kflops = kernel_flops_per_step(kname, ws_)
            launches_per_step = kd["launches"] / args.steps
            per_launch = kflops / launches_per_step if kflops and launches_per_step else None
            avg_ms = kd["ms"] / kd["launches"]
            if per_launch:
                achieved = per_launch / (avg_ms * 1e-3) / 1e12
                roof = {"bound": "tensor", "kernel": kname, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                        "frac": achieved / peak, "peak_kind": peak_kind,
                        "frac_of_measured_burst_peak": achieved / pk["bf16_tflops"],
                        "frac_of_measured_sustained_peak": achieved / pk["bf16_tflops_sustained"],
                        "frac_of_spec_peak": achieved / SPEC_BF16_TFLOPS,
                        "flops_per_launch": per_launch, "avg_launch_ms": avg_ms,
                        "timing": "CUDA events around each launch on its stream, in a second pass of the same "
                                  "steps right after the headline timing",
                        "traffic": traffic_from_profiles(kname, owner_workload(kname, ws_))}
        # the kernel pass ran the same steps as the timed region, and every
        # launch of a step is one of this library's kernels
        gpu_launches = int(sum(k["launches"] for k in kernels.values()))
        per_kernel = {k: {"launches_per_step": v["launches"] / args.steps, "ms_per_step": v["ms"] / args.steps,
                          "tflops": (kernel_flops_per_step(k, ws_) / (v["ms"] / args.steps * 1e-3) / 1e12)
                          if kernel_flops_per_step(k, ws_) else None}
                      for k, v in sorted(kernels.items(), key=lambda kv: -kv[1]["ms"])}

    # ---------------- end to end: pinned host inputs -> device, the step, loss -> host
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, job, ws_, dev, stream, barrier, ws, mlp_fl + ce_fl,
                      clocks=(lambda: ClockSampler(dev)) if not args.no_clocks else None)

    # ---------------- CPU oracle baseline (rank 0 at N = 1 only)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        tokens = CPU_SAMPLE_TOKENS_JOB.get(name) or {ws_[0].name: CPU_SAMPLE_TOKENS[name]}
        samples = [(w, oracle_sample(w, st.mi, st.ci, tokens[w.name], st.ai)) for w, st in zip(ws_, job.steps)]
        t0 = time.perf_counter()
        for w, s in samples:
            oracle_step(w, s)
        sec = time.perf_counter() - t0
        cpu = {"value": sample_work(ws_, tokens) / sec / 1e12, "unit": UNIT, "cores": oracle.num_threads(),
               "kind": "oracle",
               "sample": f"{sample_text(ws_, tokens)} through the full step at full widths; {sec:.1f} s; "
                         f"same FLOP-per-token convention as value"}

    if rank != 0:
        return 0
    in_bytes = sum(input_bytes(st) for st in job.steps)
    parts = fractions(ws_, parts_ms.get("mlp"), parts_ms.get("ce"), pk)
    parts["targets"] = {k: v for k, v in TARGETS.items()
                        if (k.startswith("mlp") and "mlp_tflops" in parts) or (k.startswith("ce") and "ce_tflops" in parts)}
    mhz = clk.get("sm_mhz") if clk else None
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {**job_config(name, ws_), "parallelism": f"t={ws_[0].t} shards on each GPU; dp{ws} "
                                                               f"(independent batches)",
                       "l2": f"no flush: inputs alone are {in_bytes / 1e9:.2f} GB per step, > 129 MB L2"},
            "timed_region_s": region_s,
            "parts": parts, "roofline": roof, "kernels": per_kernel, "gpu_launches": gpu_launches,
            "e2e": e2e, "cpu_baseline": cpu, "clocks": clk,
            "clock_normalised": {"sm_mhz_median": mhz, "tflops_per_ghz": value / (mhz * 1e-3)} if mhz else None,
            "context": PAGES_CONTEXT}
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def run_e2e(args, job, ws_, dev, stream, barrier, ws, work, clocks=None):
    """The same steps through the Python API with every step's inputs copied
    from pinned host memory (a second stream, double-buffered: step i+1's copy
    overlaps step i's compute) and the step's result read back."""
    host = {}
    for j, st in enumerate(job.steps):
        for tag, src in (("m", st.mi), ("c", st.ci), ("a", st.ai)):
            if src:
                for k, v in src.items():
                    if (tag, k) not in st.unused:
                        host[(j, tag, k)] = v.cpu().pin_memory()
    dev_in = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    # the result read back: the loss where the step has one, else the last block's output
    ce_steps = [st for st in job.steps if st.w.v_pad]
    res_host = torch.empty(ce_steps[-1].w.T, dtype=torch.float32).pin_memory() if ce_steps else None
    last = job.steps[-1]
    if res_host is None:
        res_host = torch.empty((last.w.T, last.w.h), dtype=torch.bfloat16).pin_memory()
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]    # set s holds its step's inputs
    consumed = [torch.cuda.Event() for _ in range(2)]  # the step that read set s has finished

    copy_events = []  # (start, end) of each step's copies in the timed run

    def issue_copy(i, timed=False):
        s_ = i % 2
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(consumed[s_])
            if timed:
                ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                ev[0].record(copy_stream)
            for k, v in host.items():
                dev_in[s_][k].copy_(v, non_blocking=True)
            if timed:
                ev[1].record(copy_stream)
                copy_events.append(ev)
            copied[s_].record(copy_stream)

    def compute(i):
        s_ = i % 2
        d = dev_in[s_]
        stream.wait_event(copied[s_])
        ins = []
        for j, st in enumerate(job.steps):
            w = st.w
            mi = {k: d[(j, "m", k)] for k in st.mi if ("m", k) not in st.unused} if w.f else None
            ci = {k: d[(j, "c", k)] for k in st.ci if ("c", k) not in st.unused} if w.v_pad else None
            ai = {k: d[(j, "a", k)] for k in st.ai} if w.n_heads else None
            ins.append((mi, ci, ai))
        job.run(ins)
        consumed[s_].record(stream)
        if ce_steps:
            res_host.copy_(ce_steps[-1].co["loss"], non_blocking=True)
        else:
            z_src = (torch.cat(last.zc) if last.w.sp else last.fo["Z"]) if last.w.f else last.ao["Z"]
            res_host.copy_(z_src, non_blocking=True)

    def e2e_run(n, start_event=None):
        timed = start_event is not None
        if timed:
            copy_stream.wait_event(start_event)  # the first copy starts inside the timed region
        issue_copy(0, timed)
        for i in range(n):
            if i + 1 < n:
                issue_copy(i + 1, timed)
            compute(i)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    sampler = clocks() if clocks else None
    a.record(stream)
    t_host = time.perf_counter()
    e2e_run(args.steps, a)
    host_ms = (time.perf_counter() - t_host) * 1e3  # the host's time to enqueue every step
    b.record(stream)
    torch.cuda.synchronize()
    clk = sampler.stop() if sampler else None
    barrier()
    e_ms = max_over_ranks(a.elapsed_time(b), ws, dev)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = res_host.numel() * res_host.element_size()
    copy_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in copy_events) if copy_events else None
    return {"value": job_rate(ws, work, e_ms / args.steps * 1e-3) / 1e12, "unit": UNIT,
            "ms_per_step": e_ms / args.steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "clocks": clk,
            "h2d_ms_per_step": copy_ms,
            "host_enqueue_ms_per_step": host_ms / args.steps,
            "pinned": all(v.is_pinned() for v in host.values()),
            "h2d_gb_per_s": h2d / copy_ms / 1e6 if copy_ms else None,
            "path": "vocab_ce_gb300 Python API -> C ABI; every step's inputs copied from pinned host memory "
                    "(on a second stream, double-buffered: step i+1's copy overlaps step i's compute; the first "
                    "copy and the last result read are inside the timed region)"}


def kernel_flops_one(name, w):
    T, h, f, vp = w.T, w.h, w.f, w.v_pad
    table = {}
    if f and w.act == "swiglu":
        table.update({"swiglu_fwd_gemm1_gate_up": 4.0 * T * h * f, "swiglu_fwd_gemm2_shard_sum": 2.0 * T * f * h,
                      "swiglu_bwd_dY_swiglu_grad": 2.0 * T * h * f, "swiglu_bwd_dW2": 2.0 * T * f * h,
                      "swiglu_bwd_dW1": 4.0 * T * h * f, "swiglu_bwd_dX_shard_sum": 4.0 * T * f * h})
    elif f:
        table.update({"mlp_fwd_gemm1_bias_gelu": 2.0 * T * h * f, "mlp_fwd_gemm2_shard_sum": 2.0 * T * f * h,
                      "mlp_bwd_dY_gelu_grad": 2.0 * T * h * f, "mlp_bwd_dB": 2.0 * T * f * h,
                      "mlp_bwd_dA": 2.0 * T * h * f, "mlp_bwd_dX_shard_sum": 2.0 * T * f * h})
    if vp:
        table.update({"ce_fwd_logits_stats": 2.0 * T * h * vp})
        if w.ce_grads:
            table.update({"ce_bwd_logits_dl": 2.0 * T * h * vp, "ce_bwd_dE": 2.0 * T * h * vp,
                          "ce_bwd_dH_shard_sum": 2.0 * T * h * vp})
    if w.n_heads:
        nqkv = (w.n_heads + 2 * w.n_kv_heads) * w.head_dim
        hq = w.n_heads * w.head_dim
        for k in ("attn_qkv_fwd", "attn_qkv_bwd_dX_shard_sum", "attn_qkv_bwd_dW"):
            table[k] = 2.0 * T * h * nqkv
        for k in ("attn_out_fwd_shard_sum", "attn_out_bwd_dO", "attn_out_bwd_dW"):
            table[k] = 2.0 * T * hq * h
    return table.get(name)


def owner_workload(name, ws_):
    """The name of the workload of a job whose step launches kernel `name`."""
    return next((w.name for w in ws_ if kernel_flops_one(name, w)), ws_[0].name)


def kernel_flops_per_step(name, ws_):
    """FLOPs one step spends in the kernel `name` (None for the side kernels)."""
    vals = [kernel_flops_one(name, w) for w in ws_]
    vals = [v for v in vals if v]
    return sum(vals) if vals else None


def main(argv=None):
    args = parse_args(argv)
    name = args.workload
    arm = run_reference if args.impl == "reference" else run_ours
    if name == "sweep":
        import dataclasses

        rc = 0
        for t in wl.SWEEP_T:
            w = wl.sweep_workload(t)
            if args.tokens:
                w = dataclasses.replace(w, T=args.tokens, b=1, s=args.tokens)
            rc |= arm(args, [w], name)
        return rc
    return arm(args, job_workloads(name, args.tokens), name)


if __name__ == "__main__":
    sys.exit(main())
