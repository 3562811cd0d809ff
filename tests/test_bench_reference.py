"""bench.py's reference arm (the CPU oracle) prints the contract's JSON line; CPU only."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3",
           "--ref-step-s", "0.2"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, res.stdout
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["unit"] == "tokens/s" and j["higher_is_better"] is True
    assert j["steps"] == 2 and j["warmup"] == 3 and j["n_gpus"] == 1 and j["value"] > 0
    assert j["config"]["workload"] == "tiny" and j["config"]["T"] == 64
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == j["value"] and cb["cores"] >= 1 and "passes" in cb["sample"]
    e2e = j["e2e"]
    assert e2e["value"] == j["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
