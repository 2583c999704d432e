"""Host-side checks of bench.py: workload-name parsing and the reference arm (the fp64 oracle on the
host cores) printing one JSON line in the metric and unit of the GPU arm's workload."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_paged_prefill_workload_names():
    import bench
    from attn_fwd_02_gb300 import workloads
    assert bench.paged_prefill_shape("prefill_paged") is workloads.PAGED_PREFILL
    assert bench.paged_prefill_shape("prefill_paged_fp8") is workloads.PAGED_PREFILL
    for d in (32, 64, 80, 96):
        assert bench.paged_prefill_shape(f"prefill_paged_d{d}") is workloads.PAGED_PREFILL_BY_DIM[d]
        assert bench.paged_prefill_shape(f"prefill_paged_d{d}_fp8").d == d


def run_reference(workload):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", workload,
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("workload,unit", [("prefill_paged_d32_fp8", "TFLOP/s"), ("decode_d32", "GB/s")])
def test_reference_arm_line(workload, unit):
    line = run_reference(workload)
    assert line["impl"] == "reference" and line["unit"] == unit and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert str(32) in line["config"]["workload"]
