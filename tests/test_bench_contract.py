"""The bench's JSON-line contract, on the CPU: the reference arm (the oracle
timed on the host cores) prints one line with the keys the contract names,
and the measured arm refuses to run without a CUDA device instead of falling
back to any CPU path."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout=600):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                          text=True, timeout=timeout)


def test_reference_arm_line_has_the_contract_keys():
    r = _run(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    j = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference"
    assert j["unit"] == "tok/s" and j["higher_is_better"] is True
    assert j["value"] > 0 and j["ms_per_step"] > 0
    assert j["config"]["workload"].startswith("decode_t1")
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == j["value"] and cb["sample"]
    e2e = j["e2e"]
    assert e2e["value"] == j["value"] and e2e["unit"] == j["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a CUDA device")
def test_measured_arm_refuses_without_a_gpu():
    r = _run(["--steps", "1", "--warmup", "0"], timeout=300)
    assert r.returncode != 0
    assert "no CUDA device" in (r.stdout + r.stderr)
    assert not any(ln.startswith("{") for ln in r.stdout.splitlines())
