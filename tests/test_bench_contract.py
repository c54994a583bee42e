"""The JSON line of bench.py's reference arm, on the host cores.

`bench.py --impl reference` times the fp64 oracle as the reference arm. Its
one JSON line carries the same metric, unit and configuration keys as the
GPU arm, and describes the oracle sample it timed. An end-to-end entry has
no host copies.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_reference(*extra):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *extra],
                         cwd=ROOT, capture_output=True, text=True, timeout=600, check=True).stdout
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out
    return json.loads(lines[0])


def test_reference_arm_json_line():
    d = run_reference("--config", "tiny", "--steps", "2", "--warmup", "1")
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["steps"] == 2 and d["n_gpus"] == 1 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["unit"] == "TFLOPS"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("tiny")


def test_reference_arm_on_a_packed_batch():
    d = run_reference("--config", "varlen", "--steps", "1", "--warmup", "1")
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["config"]["workload"].startswith("varlen")
