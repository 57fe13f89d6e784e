"""The benchmark's reference arm (the fp64 oracle timed on the host cores)
runs without a GPU: its one JSON line carries the keys the contract asks for,
on the same metric, unit and workload as the GPU arm, with exactly the steps
asked for and the oracle's rate as value, cpu_baseline and e2e alike."""
import importlib.util
import json
import subprocess
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parent.parent


def _bench_module():
    spec = importlib.util.spec_from_file_location("bench_for_cpu_test", ROOT / "bench.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_reference_arm_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    bench = _bench_module()
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] >= 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    cpu, e2e = d["cpu_baseline"], d["e2e"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["sample"] and cpu["value"] == d["value"]
    assert e2e == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "B=64" in d["config"]["workload"]
