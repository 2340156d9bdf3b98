"""The bench's host-side reporting on the CPU: the percentile it reports and the reference arm's
JSON line (the oracle timed on the host, rank 0 of a single process)."""
import json
import os
import random
import statistics
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_p90_is_the_nearest_rank_and_never_below_the_median():
    assert bench.p90([5.0]) == 5.0
    assert bench.p90([1.0, 2.0]) == 2.0
    assert bench.p90(list(range(10))) == 8          # 9 of 10 samples at or below it
    assert bench.p90(list(range(100))) == 89
    rng = random.Random(3)
    for n in range(1, 60):
        xs = sorted(rng.random() for _ in range(n))
        v = bench.p90(xs)
        assert v >= statistics.median(xs)
        assert sum(x <= v for x in xs) >= 0.9 * n
        assert sum(x < v for x in xs) < 0.9 * n


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    out = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in out, key
    assert out["impl"] == "reference" and out["metric"] == bench.METRIC
    assert out["steps"] == 3 and out["warmup"] == 3 and out["n_gpus"] == 1
    assert out["value"] > 0 and out["unit"] == "GB/s" and out["higher_is_better"] is True
    assert out["us_per_call"]["p90"] >= out["us_per_call"]["median"] > 0
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == out["value"] and cb["sample"]
    assert out["e2e"] == {"value": out["value"], "unit": out["unit"], "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
    assert out["config"] == bench.workload_config(bench.HEADLINE, 1)   # the device arm's config, exactly
    assert str(bench.DEFAULT["N"]) in cb["sample"] and "whole" in cb["sample"]


def test_oracle_on_cores_equals_one_whole_oracle_call():
    import numpy as np

    import oracle
    import synth

    x, xs, W, ws = synth.w8a8_inputs(5, 256, 200, seed=8, dist="mlp")
    par = bench.OracleOnCores(x, xs, W, ws, threads=4)
    try:
        np.testing.assert_array_equal(par.call(), oracle.w8a8_gemm(x, xs, W, ws))
    finally:
        par.close()


def test_device_arm_fails_loudly_without_a_gpu():
    # No CPU fallback: on a host without CUDA the default (device) arm exits non-zero and prints no
    # result line.
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "1", "--warmup", "3"], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert not [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]


def test_profile_summaries_quote_commands_the_bench_accepts():
    # Every bench command a committed ncu summary gives must still parse with the current options,
    # so that the summary can be reproduced from committed files.
    import re
    import shlex

    prof = os.path.join(ROOT, "profiles")
    found = 0
    for name in sorted(os.listdir(prof)):
        with open(os.path.join(prof, name)) as f:
            text = f.read()
        for cmd in re.findall(r"python bench\.py([^`|&>\n\\]*)", text):
            bench.build_parser().parse_args(shlex.split(cmd))
            found += 1
    assert found > 0
