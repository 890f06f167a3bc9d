"""bench.py's reference arm on the host (the fp64 oracle), on the tiny workload: one JSON
line with the fields the measurement contract asks of it."""
import json
import os
import subprocess
import sys

from conftest import ROOT


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny-fp32", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference"
    assert out["unit"] == "passes/s" and out["higher_is_better"] is True
    assert out["value"] > 0 and out["steps"] == 2 and out["warmup"] == 1
    assert out["config"]["workload"] == "tiny-fp32"
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == out["value"] and cb["cores"] >= 1
    assert out["e2e"] == {"value": out["value"], "unit": "passes/s",
                          "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # the timing fields describe what ran: measured samples, their total inside the run
    ex = out["extrapolated"]
    assert ex["passes_timed_per_step"] == 1 and ex["passes_per_step_in_value"] == 3
    assert abs(out["ms_per_step"] * out["steps"] / 1e3 - ex["timed_s"]) < 0.01 + 0.01 * ex["timed_s"]
    # the same workload identity as the native arm's line
    assert set(out["config"]) == {"workload", "N", "B", "V", "r", "hidden", "H", "K", "topc"}
