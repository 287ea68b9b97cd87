"""Host logic of bench.py that needs no GPU: which unit a workload is
measured in (algorithmic bytes for the decode kernels, M <= 32; FLOPs for the
tcgen05 GEMM, M > 32), the algorithmic byte counts of each weight form, and
the problems the bench builds for each workload."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import workloads  # noqa: E402


def _shape(spec):
    return bench.parse_shape(spec)


def test_units_follow_the_kernel_regime():
    assert bench.part_units(_shape("32,34816,5120,64,asym"))[1:] == ("GB/s", False)
    assert bench.part_units(_shape("33,34816,5120,64,asym"))[1:] == ("TFLOP/s", True)
    w = workloads.WORKLOADS["prompt_gateup_m4096_k5120_n17408"]
    units, unit, is_flops = bench.part_units(w)
    assert (unit, is_flops) == ("TFLOP/s", True) and units == 2 * 4096 * (2 * 17408) * 5120
    w = workloads.WORKLOADS["decode_gateup_silu_m1_k5120_n17408"]
    assert bench.part_units(w) == (workloads.gateup_bytes(1, 17408, 5120, 128, True), "GB/s", False)


def test_algorithmic_bytes_per_form():
    N, K, G = 256, 512, 64
    base = N * K // 2 + N * (K // G) * 2           # codes + scales
    assert workloads.algorithmic_bytes(0, N, K, G, True) == base
    assert workloads.algorithmic_bytes(0, N, K, G, False) == base + N * (K // G) // 2   # + zeros
    assert workloads.algorithmic_bytes(0, N, K, G, False, affine=True) == base + N * (K // G) * 2  # + biases
    assert workloads.algorithmic_bytes(3, N, K, G, True) == base + 3 * K * 2 + 3 * N * 2      # + x + y


def test_shape_workloads_and_forms():
    w = _shape("5,1024,512,128,affine")
    assert w["affine"] and not w["sym"] and w["kind"] == "gemm"
    w = _shape("5,1024,512,128,sym")
    assert w["sym"] and not w["affine"]


@pytest.mark.parametrize("name", ["affine_decode_m1_k5120_n34816", "tiny_gemv_m1_k512_n256"])
def test_bench_problems_carry_their_form(name):
    w = dict(workloads.WORKLOADS[name])
    w.update(N=min(w["N"], 64), K=min(w["K"], 512))  # small copy of the workload's form
    p = bench.new_problem(w)
    assert p["affine"] == w["affine"]
    assert (p["zeros"] is None) == (w["sym"] or w["affine"])
    assert ("biases" in p) == w["affine"]


def test_metric_names():
    assert bench.metric_name("decode_ffn_m1") == "W4A16 GEMM eff. HBM GB/s (M=1..16)"
    assert bench.metric_name("prompt_gateup_m4096_k5120_n17408").startswith("W4A16 fused gate/up GEMM TFLOP/s")
    assert bench.metric_name("chunk_m256_k17408_n5120") == "W4A16 GEMM TFLOP/s (M>32)"


def test_oracle_step_whole_and_sampled_columns():
    probs, is_flops = bench._oracle_problems("tiny_gemv_m1_k512_n256")
    assert not is_flops
    s, units, desc = bench._oracle_step(probs, is_flops)
    assert s > 0 and desc == "whole step"
    assert units == workloads.algorithmic_bytes(1, 256, 512, 128, True)
    # a quarter of the columns, evenly spaced, through the sampled-output path
    s, units, desc = bench._oracle_step(probs, is_flops, frac=0.25)
    assert units == workloads.algorithmic_bytes(1, 64, 512, 128, True)
    assert "64 of 256 columns" in desc
    # the FLOP unit counts 2 * rows * columns * K of the sample
    probs, is_flops = bench._oracle_problems("shape:40,64,128,64,affine")
    assert is_flops
    _, units, desc = bench._oracle_step(probs, is_flops, frac=0.5)
    assert units == 2 * 16 * 32 * 128 and "16 of 40 rows x 32 of 64 columns" in desc


def test_reference_line_echoes_the_launch():
    import argparse
    args = argparse.Namespace(workload="tiny_gemv_m1_k512_n256", steps=2, warmup=3, kernel="auto", argmax=False,
                              topk=0, noalloc=False)
    assert bench.run_reference(args, 1, 2) is None  # only rank 0 works and prints
    line = bench.run_reference(args, 0, 2)
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["sample"].startswith("whole step, 2 repetition(s)")
    # the same config dict as the CUDA arm's line for the same launch
    assert line["config"] == bench.workload_config(args, 2)
    assert line["config"]["calls_per_step"] == ["tiny_gemv_m1_k512_n256"]


def test_cpu_baseline_runs_at_least_one_step():
    cb = bench.cpu_baseline("tiny_gemv_m1_k512_n256", budget_s=0.0)
    assert cb["reps"] == 1 and cb["value"] > 0 and cb["kind"] == "oracle"
