"""The reference arm of bench.py on CPU: `--impl reference` times the
oracle on the headline workload and prints one JSON line that keeps the
benchmark contract (the keys the driver reads), with a short oracle budget
so that it runs in seconds.  The arm runs on the host alone: the product
library is never loaded in its process, and its config is the very dict
the native arm reports for the same workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Runs the arm in-process, then reports whether libpa.so was ever mapped
# into it and whether the binding module was imported.
_DRIVER = r"""
import runpy, sys
sys.argv = ["bench.py", "--impl", "reference", "--steps", "3", "--warmup", "3",
            "--cpu-budget", "0.3"]
runpy.run_path("bench.py", run_name="__main__")
maps = open("/proc/self/maps").read()
print("LIBPA_MAPPED", "libpa.so" in maps)
print("BINDING_IMPORTED", "paged_kv_cache_228_gb300.pa" in sys.modules)
"""


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "-c", _DRIVER], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    assert "LIBPA_MAPPED False" in r.stdout
    assert "BINDING_IMPORTED False" in r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "e2e", "cpu_baseline",
              "ms_per_step"):
        assert k in d, k
    assert d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert 0 < d["ms_per_step"] < 1e5
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_228_gb300 import workloads as W
    assert d["config"] == bench.workload_config(W.llama31_8b())
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] == d["value"]
    assert cpu["sample"] and cpu["cpu_model"]
