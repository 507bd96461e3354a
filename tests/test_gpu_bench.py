"""bench.py on the GPU: one short run per form prints one JSON line carrying every key of the
benchmark contract, and its launch count is the timed steps times the kernels of one step."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
@pytest.mark.parametrize("workload,unit,kernels", [("c0", "TOPS", 2), ("d3", "tok/s", 1)])
def test_bench_line_contract(workload, unit, kernels):
    steps = 3
    r = subprocess.run([sys.executable, "bench.py", "--workload", workload, "--steps", str(steps), "--warmup", "3",
                        "--no-targets", "--cpu-seconds", "0.5"], cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks",
                "gpu_launches"):
        assert key in d, key
    assert d["unit"] == unit and d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == steps
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert "workload" in d["config"]
    roof = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert roof["achieved"] > 0 and roof["peak"] > 0 and abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0 and cpu["sample"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == unit
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches_per_step"] == kernels and d["gpu_launches"] == steps * kernels
