"""Backward parity: dQ, dK, dV of sum(O * dO) vs the fp64 oracle."""
import numpy as np
import pytest

from gpu_common import device, status_ok, torch
import parity

import fa_workloads as W
import io_aware_exact_15_gb300 as fa

pytestmark = pytest.mark.gpu


def run_fwd_bwd(q, k, v, do, scale, causal, dev):
    B, H, N, d = q.shape
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    assert fa.fa_forward(qd, kd, vd, o, lse, B, H, N, d, scale, causal) == fa.FA_OK
    dq, dk, dv = (torch.full_like(qd, float("nan")) for _ in range(3))
    nbytes = fa.fa_backward_workspace_size(B, H, N, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ws.fill_(0xFF)  # contents on entry must not matter
    assert fa.fa_backward(qd, kd, vd, o, dod, lse, dq, dk, dv, B, H, N, d, scale, causal, ws,
                          nbytes) == fa.FA_OK
    status_ok()
    return o.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 100, 128, 129, 255, 300, 513])
def test_backward_small_full(N, d, causal):
    dev = device()
    q, k, v, do = W.make_qkv(2, 2, N, d, seed=N * 11 + d + causal)
    scale = 1.0 / d ** 0.5
    o, lse, dq, dk, dv = run_fwd_bwd(q, k, v, do, scale, causal, dev)
    what = f"N={N} d={d} causal={causal}"
    o_ref, lse_ref = parity.oracle_forward(q, k, v, scale, causal)
    parity.check_forward(o, lse, o_ref, lse_ref, what)
    dq_r, dk_r, dv_r = parity.oracle_backward(q, k, v, do, scale, causal)
    parity.check_grad(dq, dq_r, "dQ", what)
    parity.check_grad(dk, dk_r, "dK", what)
    parity.check_grad(dv, dv_r, "dV", what)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_backward_split_entry_points(d, causal):
    # preprocess -> main -> dq_convert, called one by one, gives the
    # gradients of fa_backward
    dev = device()
    B, H, N = 2, 3, 513
    q, k, v, do = W.make_qkv(B, H, N, d, seed=5 + d + causal)
    scale = 1.0 / d ** 0.5
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    assert fa.fa_forward(qd, kd, vd, o, lse, B, H, N, d, scale, causal) == fa.FA_OK
    dq, dk, dv = (torch.full_like(qd, float("nan")) for _ in range(3))
    nbytes = fa.fa_backward_workspace_size(B, H, N, d)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=dev)
    assert fa.fa_backward_preprocess(o, dod, B, H, N, d, ws, nbytes) == fa.FA_OK
    assert fa.fa_backward_main(qd, kd, vd, dod, lse, dk, dv, B, H, N, d, scale, causal, ws,
                               nbytes) == fa.FA_OK
    assert fa.fa_backward_dq_convert(dq, B, H, N, d, scale, ws, nbytes) == fa.FA_OK
    status_ok()
    what = f"d={d} causal={causal}"
    dq_r, dk_r, dv_r = parity.oracle_backward(q, k, v, do, scale, causal)
    parity.check_grad(dq.cpu(), dq_r, "dQ", what)
    parity.check_grad(dk.cpu(), dk_r, "dK", what)
    parity.check_grad(dv.cpu(), dv_r, "dV", what)


def test_backward_single_key_closed_form():
    # N = 1: O = V, dV = dO and dQ = dK = 0 exactly
    dev = device()
    q, k, v, do = W.make_qkv(3, 2, 1, 128, seed=77)
    o, lse, dq, dk, dv = run_fwd_bwd(q, k, v, do, 0.09, False, dev)
    assert torch.equal(o, v)
    assert torch.equal(dv, do)
    assert dq.float().abs().max().item() < 1e-4 and dk.float().abs().max().item() < 1e-4


def test_backward_is_repeatable_to_tolerance():
    # dQ is summed with fp32 atomics: two runs agree to rounding, not bits
    dev = device()
    q, k, v, do = W.make_qkv(1, 2, 640, 64, seed=3)
    a = run_fwd_bwd(q, k, v, do, 0.125, True, dev)
    b = run_fwd_bwd(q, k, v, do, 0.125, True, dev)
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])  # dK, dV: no atomics
    assert (a[2].float() - b[2].float()).abs().max().item() < 1e-2


@pytest.mark.parametrize("name", ["bert_large", "gpt2_causal"])
def test_backward_named_workload_full(name):
    dev = device()
    w = W.WORKLOADS[name]
    q, k, v, do, _ = W.make_inputs(w)
    o, lse, dq, dk, dv = run_fwd_bwd(q, k, v, do, w.scale, w.causal, dev)
    dq_r, dk_r, dv_r = parity.oracle_backward(q, k, v, do, w.scale, w.causal)
    parity.check_grad(dq, dq_r, "dQ", name)
    parity.check_grad(dk, dk_r, "dK", name)
    parity.check_grad(dv, dv_r, "dV", name)
