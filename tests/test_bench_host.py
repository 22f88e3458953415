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
    r = bench.cpu_baseline(W.WORKLOADS["single_head_fwd"], budget_s=0.5, single_thread_s=0.3)
    assert set(r) == {"value", "unit", "cores", "kind", "sample", "single_thread"}
    assert r["kind"] == "oracle" and r["unit"] == "TFLOP/s"
    assert r["cores"] == (os.cpu_count() or 1)
    assert r["value"] > 0
    # one slice, finished well inside the budget: repeated whole passes
    assert "1 of 1" in r["sample"] and "pass(es)" in r["sample"]
    st = r["single_thread"]
    assert st["cores"] == 1 and st["value"] > 0 and st["workload"] == "bert_large"
    assert "of 128 (batch, head) slices of bert_large on one thread" in st["sample"]


def test_calibration_stays_within_the_workload():
    calls = []

    def sample(n, nthreads):
        calls.append(n)

    n, (n_last, dt_last) = bench.calibrate_units(sample, 7, 1, 0.05)
    assert 1 <= n <= 7 and all(1 <= c <= 7 for c in calls)
    assert n_last == calls[-1] and dt_last >= 0


def test_compulsory_bytes_of_the_backward():
    # B1 H16 N16384 d128: Q, dO, K, V read, dK, dV written (bf16), lse and
    # D read (fp32), the fp32 dQ accumulator read and written once
    rows = 16 * 16384
    got = bench.bwd_compulsory_bytes(rows, rows, 128)
    assert got == rows * (6 * 128 * 2 + 2 * 4 + 2 * 4 * 128)
    # grouped K/V: key/value rows are a quarter of the query rows
    assert bench.bwd_compulsory_bytes(rows, rows // 4, 128) < got
    # the deterministic pass writes bf16 dQ instead of touching fp32
    assert bench.bwd_compulsory_bytes(rows, rows, 128, True) < got


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


def test_tile_model_kv_bytes():
    # dense: every CTA streams all nT key tiles (K and V, 128 x d bf16 each)
    tile = 2 * 128 * 64 * 2
    assert bench.tile_model_kv_bytes(1, 1, 512, 64, 256, False) == 2 * 4 * tile
    assert bench.tile_model_kv_bytes(1, 1, 512, 64, 128, False) == 4 * 4 * tile
    # causal, 128-row CTAs: 1 + 2 + 3 + 4 tiles; 256-row CTAs: 2 + 4
    assert bench.tile_model_kv_bytes(1, 1, 512, 64, 128, True) == 10 * tile
    assert bench.tile_model_kv_bytes(1, 1, 512, 64, 256, True) == 6 * tile
    # ragged: N = 300 has 3 tiles; the last 256-row CTA reaches tile 2 only
    assert bench.tile_model_kv_bytes(1, 1, 300, 64, 256, True) == (2 + 3) * tile
