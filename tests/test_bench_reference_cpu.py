"""The benchmark's reference arm (the CPU oracle timed on the host cores)
runs without a GPU and prints one JSON line with the contract's keys."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "1",
                        "--cpu-units", "2", "--workload", "llama31_8b_16k"], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.strip().splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert "logical CPUs" in d["cpu_baseline"]["cpu"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] == "llama31_8b_16k" and d["unit"] == "GB/s"
    # the GPU arm's compact config, key for key (the same workload, layers and timing method named)
    assert set(d["config"]) == {"workload", "batch_per_gpu", "heads", "n_tokens", "budget_tokens", "levels",
                                "parallelism", "gather", "l2", "graph", "workspace"}
    assert d["config"]["heads"] == "32/8" and d["config"]["parallelism"] == "dp1"
    assert d["config"]["l2"].startswith("2 layers rotated")
