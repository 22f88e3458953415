"""Host-side pieces of bench.py's JSON line, checked without a GPU: the
cpu_baseline object (the oracle timed on a bounded sample), the DRAM
traffic lookup that is valid only for the kernel source it was taken on,
and the sizing of the oracle sample."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import fa_workloads as W  # noqa: E402


def test_cpu_baseline_object_on_a_short_budget():
    r = bench.cpu_baseline(W.WORKLOADS["single_head_fwd"], budget_s=0.5)
    assert set(r) == {"value", "unit", "cores", "kind", "sample"}
    assert r["kind"] == "oracle" and r["unit"] == "TFLOP/s"
    assert r["cores"] == (os.cpu_count() or 1)
    assert r["value"] > 0
    # one slice, finished well inside the budget: repeated whole passes
    assert "1 of 1" in r["sample"] and "pass(es)" in r["sample"]


def test_calibration_stays_within_the_workload():
    calls = []

    def sample(n, nthreads):
        calls.append(n)

    n = bench.calibrate_units(sample, 7, 1, 0.05)
    assert 1 <= n <= 7 and all(1 <= c <= 7 for c in calls)


def test_traffic_record_needs_the_current_kernel_source():
    h = bench.kernel_source_hash(["fa_bwd.cu", "fa_ptx.cuh", "fa_sched.cuh"])
    got = bench.ncu_traffic("fa_bwd_kernel:bert_large", h)
    assert got is None or got > 0
    assert bench.ncu_traffic("fa_bwd_kernel:bert_large", "0" * 12) is None
    assert bench.ncu_traffic("no_such_kernel:bert_large", h) is None


@pytest.mark.parametrize("name", ["bert_large", "gqa_causal_n4096_d128", "bert_large_varlen"])
def test_oracle_job_units_and_flops(name):
    w = W.WORKLOADS[name]
    _, total, per_unit = bench.oracle_job(w)
    heads = w.H if w.varlen else w.B * w.H
    assert total == heads
    assert per_unit * total == pytest.approx(W.fwd_bwd_flops(w))
