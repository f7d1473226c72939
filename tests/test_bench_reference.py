"""bench.py's reference arm (the oracle on the host cores) prints one JSON line
with the keys of the benchmark contract, on CPU (no GPU needed)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e")


def _run(*extra):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2", "--warmup", "3",
           "--cpu-seconds", "5", *extra]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def _check(line, unit, higher):
    for k in KEYS:
        assert k in line, k
    assert line["impl"] == "reference" and line["unit"] == unit and line["higher_is_better"] is higher
    assert line["value"] > 0 and line["n_gpus"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"] == line["e2e"]["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_gemv_sweep():
    line = _run()
    _check(line, "GB/s", True)
    assert "qwen3-32b" in line["config"]["workload"]


@pytest.mark.parametrize("extra,tag", [((), None), (("--top-p", "0.95", "--threshold", "window"), "top-p 0.95")])
def test_reference_arm_sampler(extra, tag):
    line = _run("--workload", "reset-sampler", *extra)
    _check(line, "us/step", False)
    if tag:
        assert tag in line["config"]["workload"] and "window threshold" in line["config"]["workload"]
