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


def test_unknown_per_workload_is_rejected():
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3",
           "--per-workload", "mixtral_t512,no_such_layer"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert res.returncode == 2 and "no_such_layer" in res.stderr


def test_result_line_fields():
    """The JSON fields of one workload's measurement, assembled from a run's numbers (no GPU)."""
    sys.path.insert(0, ROOT)
    import bench
    from mixture_experts_grouped_fp32_gb300.workloads import WORKLOADS
    w = WORKLOADS["mixtral_t4096"]
    lw = bench.layer_work(w, 8)
    r = {"ms": 2.0, "steps": 20, "tokens_per_rank": w.T, "t_wall": 0.05, "clocks": None,
         "stage_ms": {"route": 0.01, "permute": 0.03, "gateup_swiglu": 1.2, "down": 0.6, "combine": 0.03},
         "staged_step_ms": 1.9, "e2e_ms": 2.1, "e2e_api": "x", "roofline": {"frac": 0.8}, "layer": lw,
         "layer_roof_ms": 1.5, "n_active": 8, "max_load": 1074, "step_ms_p10_p90": (1.9, 2.1),
         "peak_src": "measured", "ksplit": 1, "launches_per_step": 5}

    class A:
        warmup, dtype, seed, flush_l2 = 5, "bf16", 0, False
    line = bench.result_line(r, w, A(), 2)
    assert line["value"] == round(2 * 4096 / 2e-3, 2) and line["n_gpus"] == 2 and line["steps"] == 20
    assert line["layer_roofline"]["frac"] == 0.75 and line["gpu_launches"] == 100
    assert line["e2e"]["h2d_bytes_per_step"] == 4096 * 4096 * 2 + 4096 * 8 * 4
    assert line["config"]["workload"] == "mixtral_t4096" and line["higher_is_better"] is True
    assert lw["flops"] == 6 * 4096 * 2 * 4096 * 14336
