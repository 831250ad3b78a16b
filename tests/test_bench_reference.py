"""bench.py's reference arm (the float64 oracle on the host) runs on CPU for
every step kind the bench offers: one-token decode, multi-token steps and an
8-bit cache; it prints one JSON line with the contract's keys."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "3", *args], capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


@pytest.mark.parametrize("args", [
    ("--workload", "gqa_tiny"),
    ("--workload", "gqa_tiny", "--q-len", "4"),
    ("--workload", "gqa_tiny", "--kv-dtype", "fp8"),
    ("--workload", "gqa_tiny", "--kv-dtype", "fp8", "--q-len", "3"),
])
def test_reference_arm_prints_one_contract_line(args):
    d = _run(*args)
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    if "--q-len" in args:
        assert "query tokens per sequence" in d["config"]["workload"]
    if "fp8" in args:
        assert d["config"]["kv_cache"].startswith("fp8")


def test_fp8_mla_reference_arm():
    # the 8-bit latent cache: one row of codes per token, key and value decoded from it
    d = _run("--workload", "mla_decode", "--batch", "1", "--kv-dtype", "fp8")
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["kv_cache"].startswith("fp8")
