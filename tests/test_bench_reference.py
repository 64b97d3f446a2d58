"""The reference arm of bench.py on CPU: `--impl reference` times the
oracle on the headline workload and prints one JSON line that keeps the
benchmark contract (the keys the driver reads), with a short oracle budget
so that it runs in seconds."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--cpu-budget", "0.3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "e2e", "cpu_baseline"):
        assert k in d, k
    assert d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "llama3.1-8b_decode_layer"
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] == d["value"]
    assert cpu["sample"] and cpu["cpu_model"]
