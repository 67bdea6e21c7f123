"""The benchmark's accounting, on the CPU: which workloads a job runs, the
FLOP conventions, the per-kernel FLOPs the roofline divides by, and the
fractions of the peaks the targets are stated against."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_headline_job_is_the_two_target_configs():
    ws = bench.job_workloads("headline")
    assert [w.name for w in ws] == ["mlp70b", "ce128k"]
    m, c = ws
    assert (m.T, m.h, m.f, m.t) == (4096, 8192, 32768, 8)
    assert (c.T, c.h, c.v_valid, c.v_pad, c.t) == (16384, 8192, 128256, 129024, 8)
    # a smaller case of the same job keeps every width
    small = bench.job_workloads("headline", tokens=512)
    assert [w.T for w in small] == [512, 512] and small[1].v_pad == 129024


def test_flop_conventions():
    m, c = bench.job_workloads("headline")
    mlp, ce = bench.job_flops([m, c])
    assert mlp == 12.0 * 4096 * 8192 * 32768          # 4 T h f forward + 8 T h f backward
    assert ce == 8.0 * 16384 * 8192 * 129024          # logits, their recompute, dE, dH over padded ids
    assert bench.ce_model_flops(c) == 6.0 * 16384 * 8192 * 128256
    # the per-kernel FLOPs of one step add up to the step's FLOPs
    names = ["mlp_fwd_gemm1_bias_gelu", "mlp_fwd_gemm2_shard_sum", "mlp_bwd_dY_gelu_grad", "mlp_bwd_dB",
             "mlp_bwd_dA", "mlp_bwd_dX_shard_sum", "ce_fwd_logits_stats", "ce_bwd_logits_dl", "ce_bwd_dE",
             "ce_bwd_dH_shard_sum"]
    assert sum(bench.kernel_flops_per_step(n, [m, c]) for n in names) == mlp + ce
    assert bench.kernel_flops_per_step("ce_combine", [m, c]) is None
    assert bench.owner_workload("ce_bwd_dE", [m, c]) == "ce128k"
    assert bench.owner_workload("mlp_bwd_dB", [m, c]) == "mlp70b"


def test_fractions_of_the_peaks():
    ws = bench.job_workloads("headline")
    pk = {"hbm_gbs": 6808.2, "bf16_tflops": 1923.5, "bf16_tflops_sustained": 1675.1}
    mlp_fl, ce_fl = bench.job_flops(ws)
    # parts that ran at exactly 60% and 50% of 2.25 PFLOP/s
    mlp_ms = mlp_fl / (0.60 * 2250e12) * 1e3
    ce_ms = ce_fl / (0.50 * 2250e12) * 1e3
    f = bench.fractions(ws, mlp_ms, ce_ms, pk)
    assert f["mlp_frac_of_spec_peak"] == pytest.approx(0.60)
    assert f["ce_frac_of_spec_roofline"] == pytest.approx(0.50)
    assert f["mlp_frac_of_measured_burst_peak"] == pytest.approx(0.60 * 2250 / 1923.5)
    assert f["ce_frac_of_measured_sustained_roofline"] == pytest.approx(0.50 * 2250 / 1675.1)
    # the CE roofline in tokens/s: the nominal peak over 8 h v_pad FLOPs per token
    assert f["ce_roofline_tokens_per_s_spec"] == pytest.approx(2250e12 / (8 * 8192 * 129024))
    assert f["ce_tokens_per_s"] / f["ce_roofline_tokens_per_s_spec"] == pytest.approx(0.50)


def test_whole_job_rate_counts_every_rank():
    assert bench.job_rate(4, 2.0, 0.5) == 16.0


def test_traffic_is_keyed_to_each_kernels_sources(tmp_path, monkeypatch):
    # every kernel of the library maps to the translation unit its launch is compiled in
    csrc = os.path.join(ROOT, "vocab_ce_gb300", "csrc")
    units = {u for _, u in bench.KERNEL_UNITS}
    assert units <= set(os.listdir(csrc))
    ce, mlp = bench.kernel_source_hash("ce_bwd_logits_dl"), bench.kernel_source_hash("mlp_bwd_dA")
    assert ce == bench.kernel_source_hash("ce_fwd_logits_stats") and ce != mlp
    assert bench.kernel_source_hash("transpose_bf16") not in (ce, mlp)
    assert len({ce, mlp, bench.kernel_source_hash()}) == 3
    # a recorded line is used only while its kernel's sources are unchanged
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "t.md").write_text(f"    traffic_per_launch kernel=ce_bwd_logits_dl workload=ce128k bytes=1234 source={ce}\n"
                               f"    traffic_per_launch kernel=mlp_bwd_dA workload=mlp70b bytes=99 source=0000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "vocab_ce_gb300").symlink_to(os.path.join(ROOT, "vocab_ce_gb300"))
    assert bench.traffic_from_profiles("ce_bwd_logits_dl", "ce128k") == 1234
    assert bench.traffic_from_profiles("ce_bwd_logits_dl", "gpt8b") is None
    assert bench.traffic_from_profiles("mlp_bwd_dA", "mlp70b") is None


def test_source_hash_ignores_comments_only():
    code = "int f(int x) { return x + 1; }  // one\n/* two\n three */ int g;"
    assert bench._code_only(code) == bench._code_only("int f(int x) {\n  return x + 1;\n}\n// other words\nint g;")
    assert bench._code_only(code) != bench._code_only(code.replace("x + 1", "x + 2"))
