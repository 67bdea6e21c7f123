"""The multi-GPU path of the benchmark on CPU ranks (gloo, world size 2): each
rank runs its own independent batch, so the only cross-rank steps are the
barrier, the max over ranks of the timed region, and the whole-job rate
(the work of all ranks over the slowest rank's time); rank 0 alone prints.
Run as real processes, rendezvous on 127.0.0.1.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        # every rank timed its own batch: 10 ms on rank 0, 13 ms on rank 1
        ms = bench.max_over_ranks(10.0 + 3.0 * rank, ws, "cpu")
        rate = bench.job_rate(ws, 1.0e12, ms * 1e-3)
        dist.barrier()
        q.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_with_two_gloo_ranks():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(ws))
    # both ranks hold the slowest rank's time, and the job's rate counts both ranks' work
    assert [r[1] for r in res] == [13.0, 13.0]
    for _, _, rate in res:
        assert rate == pytest.approx(2 * 1.0e12 / 13.0e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench.job_rate(1, 3.0, 2.0) == 1.5


def test_reference_arm_under_torchrun_prints_once():
    # the reference arm (the CPU oracle) under a two-process launch: rank 0
    # times it and prints one JSON line; rank 1 exits 0 without work
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "attn70b", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="4")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
