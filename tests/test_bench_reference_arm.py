"""The bench's reference arm (the float64 oracle timed on the host cores) on
CPU: its JSON line keeps the contract (one line, impl "reference", the same
metric/config as the GPU arm, a cpu_baseline describing the run, an e2e with
zero host-device bytes), and the timing helpers behave."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run("--impl", "reference", "--workload", "layernorm_256", "--steps", "2", "--warmup", "0",
             "--ref-step-seconds", "0.2")
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["n_gpus"] == 1 and d["dtype"] == "f64"
    assert d["config"]["workload"] == "layernorm_256" and d["config"]["M"] == 256
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_column_workload_samples_columns():
    d = _run("--impl", "reference", "--workload", "column_layernorm", "--steps", "1", "--warmup", "0",
             "--ref-step-seconds", "0.5")
    assert d["config"]["axis"] == "col"
    assert "columns" in d["cpu_baseline"]["sample"]


def test_percentile_helper():
    sys.path.insert(0, ROOT)
    import bench
    xs = [0.9, 0.1, 0.5, 0.3, 0.7]
    assert bench.percentile(xs, 0.0) == 0.1 and bench.percentile(xs, 1.0) == 0.9
    assert bench.percentile(xs, 0.5) == 0.5
