"""bench.py --impl reference (the oracle on the host cores): one JSON line in
the same contract as the GPU arm, with the workload's shape keys in
`config`, a cpu_baseline describing the run and a zero-copy e2e object."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [x for x in out.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,unit", [("tiny", "TFLOP/s"), ("pack", "GB/s"), ("qwen", "TFLOP/s")])
def test_reference_line(workload, unit):
    d = _line("--workload", workload, "--steps", "1", "--warmup", "1", "--ref-rows", "8")
    assert d["impl"] == "reference" and d["unit"] == unit and d["value"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 1
    c = d["config"]
    for key in ("workload", "B", "S", "H", "D", "U", "A", "joint", "virtual_ranks"):
        assert key in c, key
    assert c["workload"] == workload and c["virtual_ranks"] == c["U"] * c["A"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
