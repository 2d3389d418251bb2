"""bench.py's command line on CPU: the reference arm (the oracle timed on the host) prints one
JSON line with every key the benchmark contract names, for a decode and a prefill workload,
and the argument checks refuse what the contract forbids (fewer than 3 warm-up steps)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e")


def _bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    return r


@pytest.mark.parametrize("workload,unit", [("tiny", "GB/s"), ("prefill_tiny", "TFLOP/s")])
def test_reference_arm_prints_the_contract_line(workload, unit):
    r = _bench("--impl", "reference", "--workload", workload, "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in KEYS:
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == unit and d["n_gpus"] == 1
    assert d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == workload
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0


def test_too_few_warmup_steps_are_refused():
    r = _bench("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "2")
    assert r.returncode != 0
    assert "warmup" in r.stderr
