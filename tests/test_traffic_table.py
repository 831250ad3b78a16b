"""The DRAM traffic table that bench.py reports as roofline.traffic
(profiles/traffic.json): every entry names a kernel of the source file it
was measured on, points at the profile summary that records the capture, and,
for the workloads whose contexts are fixed, stays within a few percent of the
unique KV bytes of a step (each cached token is read once; more would be
re-reads). Entries whose source hash no longer matches are reported null by
bench.py, which is checked too."""
import hashlib
import json
import os
import re

import pytest

import bench
from sequence_sharded_decode_gb300 import configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "profiles", "traffic.json")
SRC = {"mla": "dcp_mla.cu", "gqa": "dcp_gqa.cu"}


def _entries():
    with open(TABLE) as f:
        return json.load(f)


def _src_file(workload: str) -> str:
    return SRC[workload.split("_")[0]]


@pytest.mark.parametrize("workload", sorted(_entries()))
def test_entry_is_complete(workload):
    e = _entries()[workload]
    assert re.fullmatch(r"[0-9a-f]{16}", e["source_sha256_16"])
    assert e["dram_bytes_per_launch"] > 0
    assert os.path.isfile(os.path.join(ROOT, e["summary"])), e["summary"]
    src = open(os.path.join(ROOT, "sequence_sharded_decode_gb300", "csrc", _src_file(workload))).read()
    assert re.search(r"\b" + e["kernel"] + r"\s*\(", src), f"{e['kernel']} is not a kernel of {_src_file(workload)}"
    assert "ncu" in e["how"] and "dram__bytes_read.sum" in e["how"]


@pytest.mark.parametrize("workload,kv_dtype", [("mla_long", "bf16"), ("gqa_mid", "bf16"),
                                               ("mla_long", "fp8"), ("gqa_mid", "fp8")])
def test_fixed_context_traffic_is_the_kv_once(workload, kv_dtype):
    name = workload + ("_fp8" if kv_dtype == "fp8" else "")
    e = _entries()[name]
    wl = configs.get(workload).with_(kv_dtype=kv_dtype)
    # every sequence attends its ctx_fixed cached tokens plus the step's new one
    kv = int(wl.batch) * (int(wl.ctx_fixed) + 1) * wl.kv_bytes_per_token
    ratio = e["dram_bytes_per_launch"] / kv
    assert 1.0 <= ratio <= 1.05, f"{name}: DRAM bytes {ratio:.3f} x the unique KV bytes"


@pytest.mark.parametrize("workload", sorted(_entries()))
def test_bench_reports_an_entry_only_for_its_current_source(workload):
    e = _entries()[workload]
    src = os.path.join(ROOT, "sequence_sharded_decode_gb300", "csrc", _src_file(workload))
    current = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] == e["source_sha256_16"]
    got = bench._traffic_for(_src_file(workload), workload)
    assert got == (float(e["dram_bytes_per_launch"]) if current else None)
