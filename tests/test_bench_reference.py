"""The benchmark's reference arm (the fp64 oracle timed on the host cores)
prints one JSON line with the contract's keys, for every op, on CPU."""

from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("op", ["verify", "draft_sample", "greedy", "topk", "topp", "lmhead"])
def test_reference_arm_prints_the_contract_line(op):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--op", op,
                        "--config", "c1", "--steps", "2", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "cpu_baseline", "e2e", "config"):
        assert key in d, key
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
