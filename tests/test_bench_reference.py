"""The reference arm of the benchmark (the oracle timed on the host cores)
prints one JSON line with the contract's keys, on CPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e")


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "0", "--steps", "3",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert all(k in d for k in KEYS), sorted(set(KEYS) - set(d))
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["vs_baseline"] is None and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_cpu_baseline_reports_cores_and_both_thread_counts():
    """The CPU baseline times the oracle single-threaded and on all host cores
    and states the core count it found."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    wl = workloads.make(workloads.spec(0))
    kv = workloads.kv_bytes_per_token(wl.spec) * int(wl.kv_len.sum())
    cb = bench.cpu_baseline(wl, kv, budget_s=0.0, max_steps=1)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s"
    assert cb["host_cores"] == bench.cpu_threads() >= 1
    assert cb["threads"] == cb["cores"] == bench.oracle_threads()
    assert cb["single_thread"]["threads"] == 1 and cb["single_thread"]["value"] > 0
    assert cb["all_cores"]["value"] == cb["value"] > 0
