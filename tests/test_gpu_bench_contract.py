"""bench.py prints one JSON line with every key of its contract (a short run of
the fp32 toy layer)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_json_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "toy", "--steps", "3",
           "--warmup", "3", "--no-cpu-baseline",
           "--configs", "sweep_T4096_s0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e",
                "gpu_launches", "roofline", "cpu_baseline", "clocks"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["higher_is_better"] is True
    assert line["scaling"] == "weak" and line["vs_baseline"] is None
    assert line["config"]["workload"] == "toy" and line["dtype"] == "f32"
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 4096 * 512 * 4 == e2e["d2h_bytes_per_step"]
    # counted by the library: route, count, scan, place, tf32 split, up, down, combine
    assert line["gpu_launches"] == 8 * 3 and line["launches_per_step"] == 8
    rf = line["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in rf, key
    # the toy's fp32 experts run on the tensor cores (three tf32 products per product)
    assert rf["bound"] == "tensor" and rf["achieved"] > 0 and rf["peak"] > 0
    assert abs(rf["achieved"] - 3 * rf["fp32_TFLOP/s"]) < 1e-6 * rf["achieved"]
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert set(line["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    # per-kernel times come from the timed pass and add up to at most the step
    ks = line["kernels"]
    assert abs(sum(ks[n]["ms"] for n in ("route", "dispatch", "ffn", "combine"))
               - line["phase_sum_ms"]) < 1e-9
    assert line["phase_sum_ms"] <= line["ms_per_step"] * 1.0001
    lf = line["layer_forward"]
    assert lf["ms_per_step"] > 0 and set(lf["clocks"]) >= {"sm_mhz", "reasons"}
    (rec,) = line["configs"]
    assert rec["workload"] == "sweep_T4096_s0" and rec["value"] > 0 and rec["steps"] >= 20
    assert "route_permute_unpermute" in rec["kernels"] and "flushed" in rec["l2"]
    # 256 experts at T=4096: a sliced router (its slices merged inside a cluster), count, scan,
    # place, combine
    assert rec["launches_per_step"] == 5 and rec["gpu_launches"] == 5 * rec["steps"]
    assert set(rec["clocks"]) >= {"sm_mhz", "reasons"}
