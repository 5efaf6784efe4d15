"""bench.py's reference arm on the host: the oracle timed on a bounded
sample of the requested workload, with the same metric, unit and workload
name as the GPU arm (here a small layer with Zipf row degrees, as the
GPT-2-shaped MLP layers use)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line_on_a_zipf_layer():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--out", "300", "--inp", "200",
           "--sparsity", "90", "--zipf", "1.2", "--batch", "4", "--steps", "2", "--warmup", "1"]
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    d = json.loads(p.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference"
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "layer300x200_s90_zipf1.2_b4"
    assert "Zipf (s = 1.2)" in d["config"]["description"]
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
