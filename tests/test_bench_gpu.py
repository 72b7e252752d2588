"""bench.py's JSON line on a GPU (small workload): every key the line promises is
present and consistent."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_has_the_contract_keys():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "gpt2", "--steps", "2",
                        "--warmup", "3", "--no-cpu-baseline", "--no-sweep"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    b = lines[0]
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in b, k
    assert b["value"] > 0 and b["n_gpus"] == 1 and b["steps"] == 2 and b["warmup"] == 3
    assert b["higher_is_better"] is True and b["scaling"] == "weak"
    rf = b["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in rf, k
    assert rf["bound"] in ("hbm", "tensor", "alu") and 0 < rf["frac"] < 1.5
    e2e = b["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert b["gpu_launches"] >= 2 * 6                   # at least the GEMMs of two steps
    assert "sm_mhz" in b["clocks"] and "reasons" in b["clocks"]
    assert b["slope_adapters"]["ms_per_step"] > 0 and b["graphs"]["graph_ms_per_step"] > 0
    assert b["prune"]["value"] > 0
