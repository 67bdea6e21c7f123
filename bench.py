#!/usr/bin/env python
"""Benchmark: tensor-parallel MLP block forward+backward and fused
vocabulary-parallel cross-entropy forward+backward, all t shards on one GPU.

One step = one pass of the whole path over one batch of synthetic inputs
resident in HBM: tp_mlp_forward, tp_mlp_backward, vocab_parallel_ce (loss,
dH, dE). The default workload is the 8.3B-shaped block (T = 8192 tokens,
h = 3072, f = 12288, vocabulary 50,257 padded to 51,200, t = 8).

Printed (rank 0, one JSON line): whole-job TFLOP/s over the step (MLP
12 T h f + CE 8 T h v_pad FLOPs, the CE count including the logit recompute
that unmaterialised logits require), the MLP TFLOP/s and CE tokens/s parts,
the end-to-end figure through the Python API from pinned host buffers, the
roofline of the dominant kernel, SM clocks during the timed region, and the
CPU oracle timed on a bounded sample on this host.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W]
                       [--impl ours|reference]
                       [--workload gpt8b|gpt8b_chain|mlp70b|mlp70b_sp|ce128k|ce128k_eval|
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
# tokens the CPU oracle processes per timed sample
CPU_SAMPLE_TOKENS = {"gpt8b": 512, "gpt8b_chain": 512, "mlp70b": 192, "mlp70b_sp": 192, "ce128k": 96, "ce128k_eval": 256,
                     "swiglu70b": 144, "attn70b": 512, "sweep": 512}
REF_STEP_TOKENS = {"gpt8b": 8, "gpt8b_chain": 8, "mlp70b": 4, "mlp70b_sp": 4, "ce128k": 2, "ce128k_eval": 4, "swiglu70b": 3,
                   "attn70b": 8, "sweep": 8}


# ---------------------------------------------------------------------- setup
def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["gpt8b", "gpt8b_chain", "mlp70b", "mlp70b_sp", "ce128k", "ce128k_eval",
                                          "swiglu70b", "attn70b", "sweep"], default="gpt8b")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    return p.parse_args()


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


def flops(w):
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
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------- traffic from committed ncu summaries
def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("gemm.cuh", "gemm_pair.cuh", "gemm_launch.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "vocab_ce_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel, workload):
    """dram bytes per launch recorded in profiles/ for this kernel and workload,
    if the GEMM source has not changed since the capture; else None."""
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    src = kernel_source_hash()
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


def oracle_rate(w, s, n_tokens, reps=1):
    """(TFLOP/s in the bench's FLOP convention, seconds per rep)."""
    mlp, ce = flops(w)
    work = (mlp + ce) / w.T * n_tokens
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_step(w, s)
    dt = (time.perf_counter() - t0) / reps
    return work / dt / 1e12, dt


# ---------------------------------------------------------------------- arms
def run_reference(args, w, name):
    import oracle

    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    oracle.build()
    n = REF_STEP_TOKENS[name]
    mi = ((wl.swiglu_inputs if w.act == "swiglu" else wl.mlp_inputs)(w, seed=0)) if w.f else None
    ci = wl.ce_inputs(w, seed=0) if w.v_pad else None
    ai = wl.attn_inputs(w, seed=0) if w.n_heads else None
    s = oracle_sample(w, mi, ci, n, ai)
    for _ in range(args.warmup):
        oracle_step(w, s)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(w, s)
        times.append(time.perf_counter() - t0)
    dt = sum(times) / len(times)
    mlp, ce = flops(w)
    value = (mlp + ce) / w.T * n / dt / 1e12
    sample = f"first {n} of {w.T} tokens at full h, f, v per step (weights in full), fp64 oracle"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, name),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w, name):
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    import vocab_ce_gb300 as tp

    step = Step(w, dev, seed=rank)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        step.run()
    torch.cuda.synchronize()
    assert tp.device_status() == 0, "device status after warm-up"

    def barrier():
        if ws > 1:
            import torch.distributed as dist

            dist.barrier()

    # ---------------- timed region (device-resident inputs)
    mlp_fl, ce_fl = flops(w)
    segs = step.segments()
    ev = [[(part, torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for part, _ in segs]
          for _ in range(args.steps)]
    clocks = ClockSampler(dev, enabled=not args.no_clocks)
    barrier()
    torch.cuda.synchronize()
    tp.profile_enable(True)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        for (_, a, b), (_, fn) in zip(ev[i], segs):
            a.record(stream)
            fn()
            b.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    kernels = tp.profile_read()
    tp.profile_enable(False)
    clk = clocks.stop()
    assert tp.device_status() == 0, "device status after the timed region"
    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(elapsed_ms, ws, dev)
    ms_step = elapsed_ms / args.steps
    mlp_ms = sum(a.elapsed_time(b) for e in ev for part, a, b in e if part == "mlp") / args.steps
    ce_ms = sum(a.elapsed_time(b) for e in ev for part, a, b in e if part == "ce") / args.steps
    value = job_rate(ws, mlp_fl + ce_fl, ms_step * 1e-3) / 1e12

    pk, pk_src = peaks()
    # ---------------- roofline of the dominant kernel
    dominant = max(kernels.items(), key=lambda kv: kv[1]["ms"]) if kernels else None
    roof = None
    if dominant:
        kname, kd = dominant
        kflops = kernel_flops_per_step(kname, w)
        launches_per_step = kd["launches"] / args.steps
        per_launch = kflops / launches_per_step if kflops and launches_per_step else None
        avg_ms = kd["ms"] / kd["launches"]
        if per_launch:
            achieved = per_launch / (avg_ms * 1e-3) / 1e12
            roof = {"bound": "tensor", "kernel": kname, "achieved": achieved, "peak": pk["bf16_tflops_sustained"],
                    "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops_sustained"],
                    "peak_kind": f"{pk_src} sustained bf16 (kernel timed inside a long step)",
                    "frac_of_burst_peak": achieved / pk["bf16_tflops"],
                    "flops_per_launch": per_launch, "avg_launch_ms": avg_ms,
                    "traffic": traffic_from_profiles(kname, name)}
    gpu_launches = int(sum(k["launches"] for k in kernels.values()))
    per_kernel = {k: {"launches": v["launches"], "ms_per_step": v["ms"] / args.steps,
                      "tflops": (kernel_flops_per_step(k, w) / (v["ms"] / args.steps * 1e-3) / 1e12)
                      if kernel_flops_per_step(k, w) else None}
                  for k, v in sorted(kernels.items(), key=lambda kv: -kv[1]["ms"])}

    # ---------------- end to end: pinned host inputs -> device, the step, loss -> host
    e2e = None
    if not args.no_e2e:
        host = {}
        for tag, src in (("m", step.mi), ("c", step.ci), ("a", step.ai)):
            if src:
                for k, v in src.items():
                    if (tag, k) not in step.unused:
                        host[tag + k] = v.cpu().pin_memory()
        # two device copies of the inputs: step i+1's inputs are copied on a
        # second stream while step i computes from the other set
        dev_in = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
        loss_host = torch.empty(w.T, dtype=torch.float32).pin_memory() if w.v_pad else None
        z_host = torch.empty((w.T, w.h), dtype=torch.bfloat16).pin_memory() if not w.v_pad else None
        copy_stream = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event() for _ in range(2)]    # set s holds its step's inputs
        consumed = [torch.cuda.Event() for _ in range(2)]  # the step that read set s has finished

        def issue_copy(i):
            s_ = i % 2
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(consumed[s_])
                for k, v in host.items():
                    dev_in[s_][k].copy_(v, non_blocking=True)
                copied[s_].record(copy_stream)

        def compute(i):
            s_ = i % 2
            d = dev_in[s_]
            stream.wait_event(copied[s_])
            mi = {k: d["m" + k] for k in step.mi if ("m", k) not in step.unused} if w.f else None
            ci = {k: d["c" + k] for k in step.ci if ("c", k) not in step.unused} if w.v_pad else None
            ai = {k: d["a" + k] for k in step.ai} if w.n_heads else None
            step.run(mi, ci, ai)
            consumed[s_].record(stream)
            if w.v_pad:
                loss_host.copy_(step.co["loss"], non_blocking=True)
            else:
                z_src = (torch.cat(step.zc) if w.sp else step.fo["Z"]) if w.f else step.ao["Z"]
                z_host.copy_(z_src, non_blocking=True)

        def e2e_run(n, start_event=None):
            if start_event is not None:
                copy_stream.wait_event(start_event)  # the first copy starts inside the timed region
            issue_copy(0)
            for i in range(n):
                if i + 1 < n:
                    issue_copy(i + 1)
                compute(i)

        e2e_run(2)
        torch.cuda.synchronize()
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_run(args.steps, a)
        b.record(stream)
        torch.cuda.synchronize()
        barrier()
        e_ms = a.elapsed_time(b)
        e_ms = max_over_ranks(e_ms, ws, dev)
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = (loss_host.numel() * 4) if w.v_pad else z_host.numel() * 2
        e2e = {"value": job_rate(ws, mlp_fl + ce_fl, e_ms / args.steps * 1e-3) / 1e12, "unit": UNIT,
               "ms_per_step": e_ms / args.steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "path": "vocab_ce_gb300 Python API -> C ABI; every step's inputs copied from pinned host memory "
                       "(on a second stream, double-buffered: step i+1's copy overlaps step i's compute; the first "
                       "copy and the last result read are inside the timed region)"}

    # ---------------- CPU oracle baseline (rank 0 at N = 1 only)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        n = CPU_SAMPLE_TOKENS[name]
        s = oracle_sample(w, step.mi, step.ci, n, step.ai)
        rate, sec = oracle_rate(w, s, n)
        cpu = {"value": rate, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"first {n} of {w.T} tokens through the full step ({workload_config(w, name)['workload'].split(':')[0]}) "
                         f"at full widths; {sec:.1f} s; same FLOP-per-token convention as value"}

    if rank != 0:
        return 0
    ws_bytes = input_bytes(step)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {**workload_config(w, name), "parallelism": f"t={w.t} shards on each GPU; dp{ws} (independent batches)",
                       "l2": f"no flush: inputs alone are {ws_bytes / 1e9:.2f} GB per step, > 129 MB L2"},
            "parts": {"mlp_tflops": (mlp_fl / (mlp_ms * 1e-3) / 1e12) if w.f else None, "mlp_ms": mlp_ms if w.f else None,
                      "attn_proj_tflops": (mlp_fl / (mlp_ms * 1e-3) / 1e12) if w.n_heads else None,
                      "attn_proj_ms": mlp_ms if w.n_heads else None,
                      "attn_proj_frac_of_peak": ((mlp_fl / (mlp_ms * 1e-3) / 1e12) / pk["bf16_tflops_sustained"])
                      if w.n_heads else None,
                      "ce_tokens_per_s": (w.T / (ce_ms * 1e-3)) if w.v_pad else None,
                      "ce_tflops": (ce_fl / (ce_ms * 1e-3) / 1e12) if w.v_pad else None, "ce_ms": ce_ms if w.v_pad else None,
                      "mlp_frac_of_peak": ((mlp_fl / (mlp_ms * 1e-3) / 1e12) / pk["bf16_tflops_sustained"]) if w.f else None,
                      "ce_frac_of_roofline": ((ce_fl / (ce_ms * 1e-3) / 1e12) / pk["bf16_tflops_sustained"]) if w.v_pad else None},
            "roofline": roof, "kernels": per_kernel, "gpu_launches": gpu_launches,
            "e2e": e2e, "cpu_baseline": cpu, "clocks": clk}
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def kernel_flops_per_step(name, w):
    T, h, f, vp = w.T, w.h, w.f, w.v_pad
    table = {
        "mlp_fwd_gemm1_bias_gelu": 2.0 * T * h * f, "mlp_fwd_gemm2_shard_sum": 2.0 * T * f * h,
        "mlp_bwd_dY_gelu_grad": 2.0 * T * h * f, "mlp_bwd_dB": 2.0 * T * f * h, "mlp_bwd_dA": 2.0 * T * h * f,
        "mlp_bwd_dX_shard_sum": 2.0 * T * f * h,
        "swiglu_fwd_gemm1_gate_up": 4.0 * T * h * f, "swiglu_fwd_gemm2_shard_sum": 2.0 * T * f * h,
        "swiglu_bwd_dY_swiglu_grad": 2.0 * T * h * f, "swiglu_bwd_dW2": 2.0 * T * f * h,
        "swiglu_bwd_dW1": 4.0 * T * h * f, "swiglu_bwd_dX_shard_sum": 4.0 * T * f * h,
        "ce_fwd_logits_stats": 2.0 * T * h * vp, "ce_bwd_logits_dl": 2.0 * T * h * vp,
        "ce_bwd_dE": 2.0 * T * h * vp, "ce_bwd_dH_shard_sum": 2.0 * T * h * vp,
    }
    if w.n_heads:
        nqkv = (w.n_heads + 2 * w.n_kv_heads) * w.head_dim
        hq = w.n_heads * w.head_dim
        for k in ("attn_qkv_fwd", "attn_qkv_bwd_dX_shard_sum", "attn_qkv_bwd_dW"):
            table[k] = 2.0 * T * h * nqkv
        for k in ("attn_out_fwd_shard_sum", "attn_out_bwd_dO", "attn_out_bwd_dW"):
            table[k] = 2.0 * T * hq * h
    return table.get(name)


def main():
    args = parse_args()
    name = args.workload
    if name == "sweep":
        rc = 0
        for t in wl.SWEEP_T:
            rc |= (run_reference if args.impl == "reference" else run_ours)(args, wl.sweep_workload(t), name)
        return rc
    w = wl.WORKLOADS[name]
    return run_reference(args, w, name) if args.impl == "reference" else run_ours(args, w, name)


if __name__ == "__main__":
    sys.exit(main())
