"""The bench's reference arm (the oracle timed on the host cores) runs without
a GPU and prints one JSON line in the contract's form."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_contract_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
           "toy", "--steps", "3", "--warmup", "2", "--ref-budget-s", "5"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["steps"] == 3 and line["warmup"] == 2 and line["n_gpus"] == 1
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "toy"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert "measured" in cb["sample"] and cb["tokens_per_step"] >= 1
    # the reported per-step time is the time a step took (it fits in the run)
    assert line["ms_per_step"] * line["steps"] <= line["sample_wall_s"] * 1e3 * 1.05 + 1.0
    assert abs(line["value"] - cb["tokens_per_step"] / (line["ms_per_step"] / 1e3)) \
        <= 1e-6 * line["value"]
    for key in ("T", "d", "E", "k", "R", "d_ff", "act", "score", "capacity_factor", "n_shared"):
        assert key in line["config"], key
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
