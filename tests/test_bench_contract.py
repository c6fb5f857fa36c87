"""bench.py's host side, on the CPU: the JSON line of the reference arm (the float64 oracle timed
on host cores) carries every key of the benchmark contract and at least 3 warm-up steps, and the
per-kernel FLOP factors that the roofline figures use add up to the 8 N d V of a forward +
backward for every launch structure the library uses."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_json_line_has_the_contract_keys():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny-fp32", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    # fewer than 3 warm-up steps are raised to 3 (the benchmark's timing rule)
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["metric"] == bench.METRIC
    assert d["config"]["workload"] == "tiny-fp32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("kernels", [
    ("tc_fwd_lse", "tc_bwd_grad", "tc_dh_dw"),        # gradient and dW + dH launches per strip
    ("tc_fwd_lse", "tc_bwd"),                         # overlapped small backward steps
    ("simt_fwd_lse", "simt_bwd_grad", "simt_dh", "simt_dw"),  # exact fp32 on the CUDA cores
])
def test_flop_factors_add_up_to_a_forward_and_backward(kernels):
    assert sum(bench.GEMM_FLOP_FACTOR[k] for k in kernels) == 8


def test_whole_job_throughput_counts_every_rank():
    assert bench.tokens_per_second(1, 32768, 140.0) == pytest.approx(32768 / 0.140)
    assert bench.tokens_per_second(4, 32768, 140.0) == pytest.approx(4 * 32768 / 0.140)
