"""bench.py's JSON line on a GPU: one line, every key of the contract, and
numbers that hang together (the kernel is part of the step, the roofline
fraction is achieved / peak)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_bench_line_contract():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "sq4096_uniform", "--steps", "3",
           "--warmup", "3", "--no-cpu", "--no-probes", "--e2e-steps", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "sq4096_uniform" and d["config"]["path"] == "tf32x3"
    flop = 2.0 * 4096 ** 3
    assert abs(d["value"] - flop / (d["ms_per_step"] * 1e-3) / 1e12) < 1e-6 * d["value"]
    roof = d["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert roof["kernel_ms"] <= d["ms_per_step"] and roof["achieved"] >= d["value"]
    e2e = d["e2e"]
    assert e2e["h2d_bytes_per_step"] == 2 * 4 * 4096 ** 2 and e2e["d2h_bytes_per_step"] == 4 * 4096 ** 2
    assert 0 < e2e["value"] < roof["achieved"]
    assert d["gpu_launches"] >= d["steps"]
