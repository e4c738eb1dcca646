"""bench.py's reference arm (the oracle on the host cores) prints one JSON
line with the same metric, unit and workload as our arm, its CPU baseline
and an end-to-end figure with no host-device bytes; a run with fewer than
three warm-up steps is refused.  Runs on the CPU."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*extra):
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-budget", "0.3",
           *extra]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def _check_common(d):
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["data"] == "synthetic" and d["dtype"] == "f64" and d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_decode_reference_line():
    """The line for a given workload (the tiny batch: the default long-context
    batch takes minutes to synthesise on a slow host; the arm is the same)."""
    sys.path.insert(0, ROOT)
    import bench

    d = _run("--workload", "tiny_f32")
    _check_common(d)
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["config"]["workload"] == "tiny_f32"


def test_reference_arm_defaults_to_our_workload():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.DEFAULT_WORKLOAD == "long_bf16"
    src = open(os.path.join(ROOT, "bench.py")).read()
    assert 'ap.add_argument("--workload", default=DEFAULT_WORKLOAD' in src


def test_prefill_reference_line():
    d = _run("--prefill")
    _check_common(d)
    assert d["metric"] == "prefill attention TFLOP/s" and d["unit"] == "TFLOP/s"
    assert d["config"]["workload"] == "prefill_bf16" and d["config"]["new"] == 512


def test_fewer_than_three_warmup_steps_are_refused():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--warmup", "2"], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "warmup" in r.stderr
