"""The benchmark's reference arm (the CPU oracle) prints one well-formed
JSON line for every operation; run here on the CPU with a single step."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup",
        "ms_per_step", "higher_is_better", "scaling", "vs_baseline", "dtype",
        "data", "config", "cpu_baseline", "e2e", "gpu_launches"}


@pytest.mark.parametrize("op,workload", [
    ("forward", "small_4x1000"), ("backward", "small_4x1000"),
    ("attention", "attention_2x8x4096_causal"),
    ("biencoder", "biencoder_4x8x1024x256x64")])
def test_reference_arm_line(op, workload):
    res = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
         "--op", op, "--workload", workload, "--steps", "1", "--warmup", "0"],
        capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["gpu_launches"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
