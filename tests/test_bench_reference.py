"""bench.py --impl reference: the oracle arm's JSON line on the host cores.

The reference arm times the fp64 oracle on a bounded sample of the workload
the GPU arm runs; its line must describe that same workload (name, B) and
carry the keys the bench contract names. Runs on the CPU only.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _reference_line(workload):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload,
                        "--steps", "1", "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,B,name", [
    ("colbert_full", 100_000, "colbert_full_q32_nd128_d128_B100000_bf16"),
    ("pq", 500_000, "pq_m16_k256_q32_d128_B500000"),
])
def test_reference_line_names_the_gpu_arms_workload(workload, B, name):
    d = _reference_line(workload)
    assert d["impl"] == "reference"
    assert d["config"]["workload"] == name and d["config"]["B"] == B
    assert d["unit"] == "docs/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["steps"] == 1 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["e2e"] == {"value": d["value"], "unit": "docs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert "tokens" not in d["config"]          # a sample's token count is not the workload's
