"""bench.py's host logic, without a GPU: the traffic record is reported only
for the GEMM source it was taken on, the reference arm (the oracle on host
cores) prints one JSON line with the contract's keys, and the dtype names
follow each workload's arithmetic."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from workloads import WORKLOADS  # noqa: E402

GEMM_SRC = os.path.join(ROOT, "exact_modular_int8_gb300", "csrc", "gemm_tc.cu")


def test_traffic_record_follows_the_kernel_source(tmp_path):
    rec = bench.gemm_traffic_record(GEMM_SRC)
    assert rec is not None and int(rec["traffic_bytes_per_launch"]) > 0 and rec["workload"] in WORKLOADS
    changed = tmp_path / "gemm_tc.cu"
    changed.write_bytes(open(GEMM_SRC, "rb").read() + b"\n")
    assert bench.gemm_traffic_record(str(changed)) is None
    assert bench.gemm_traffic_record(str(tmp_path / "missing.cu")) is None


def test_workload_dtypes():
    want = {"int": "int64", "limbs": "int64", "normal": "f64", "interval": "f64", "normal32": "f32"}
    for w in WORKLOADS.values():
        assert bench.workload_dtype(w) == want[w.kind], w.name


@pytest.mark.timeout(300)
def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["unit"] == "TOPS" and d["config"]["workload"] == "exact24_4096"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
