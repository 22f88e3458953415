"""Deterministic backward (key-tile pass without dQ + query-tile dQ pass):
parity with the fp64 oracle, bit-identical results from run to run, and
dK, dV bit-identical to fa_backward's (same products in the same order)."""
import pytest

from gpu_common import device, status_ok, torch
import parity

import fa_workloads as W
import io_aware_exact_15_gb300 as fa
import oracle

pytestmark = pytest.mark.gpu


def forward(qd, kd, vd, scale, causal):
    B, H, N, d = qd.shape
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=qd.device)
    assert fa.fa_forward(qd, kd, vd, o, lse, B, H, N, d, scale, causal) == fa.FA_OK
    return o, lse


def backward(fn, qd, kd, vd, o, dod, lse, scale, causal, ws_bytes=None):
    B, H, N, d = qd.shape
    dq, dk, dv = (torch.full_like(qd, float("nan")) for _ in range(3))
    nbytes = ws_bytes or fa.fa_backward_workspace_size(B, H, N, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=qd.device)
    assert fn(qd, kd, vd, o, dod, lse, dq, dk, dv, B, H, N, d, scale, causal, ws,
              nbytes) == fa.FA_OK
    status_ok()
    return dq, dk, dv


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 200, 257, 384])
def test_deterministic_small_full(N, d, causal):
    dev = device()
    q, k, v, do = W.make_qkv(2, 3, N, d, seed=400 + N + d + causal)
    scale = 1.0 / d ** 0.5
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = forward(qd, kd, vd, scale, causal)
    # the smallest workspace it accepts: D only
    ws_min = (2 * 3 * N * 4 + 255) // 256 * 256
    dq, dk, dv = backward(fa.fa_backward_deterministic, qd, kd, vd, o, dod, lse, scale, causal,
                          ws_bytes=ws_min)
    what = f"N={N} d={d} causal={causal}"
    f = parity.f64
    dq_r, dk_r, dv_r = oracle.backward(f(q), f(k), f(v), f(do), scale, causal=causal)
    parity.check_grad(dq.cpu(), dq_r, "dQ", what)
    parity.check_grad(dk.cpu(), dk_r, "dK", what)
    parity.check_grad(dv.cpu(), dv_r, "dV", what)
    # dK, dV: the same products in the same order as fa_backward
    _, dk_a, dv_a = backward(fa.fa_backward, qd, kd, vd, o, dod, lse, scale, causal)
    assert torch.equal(dk, dk_a) and torch.equal(dv, dv_a)


@pytest.mark.parametrize("causal", [False, True])
def test_bit_identical_runs(causal):
    dev = device()
    B, H, N, d = 2, 8, 2048, 128
    q, k, v, do = W.make_qkv(B, H, N, d, seed=77 + causal)
    scale = 1.0 / d ** 0.5
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = forward(qd, kd, vd, scale, causal)
    runs = [backward(fa.fa_backward_deterministic, qd, kd, vd, o, dod, lse, scale, causal)
            for _ in range(3)]
    for other in runs[1:]:
        for a, b in zip(runs[0], other):
            assert torch.equal(a, b)
    # and it agrees with the atomic path within the tolerance
    ref = backward(fa.fa_backward, qd, kd, vd, o, dod, lse, scale, causal)
    parity.check_grad(runs[0][0].cpu(), parity.f64(ref[0]), "dQ", "vs fa_backward")


def test_deterministic_longseq_sampled_rows():
    dev = device()
    wl = W.WORKLOADS["longseq_causal_n4096_d128"]
    q, k, v, do, _ = W.make_inputs(wl)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = forward(qd, kd, vd, wl.scale, wl.causal)
    dq, dk, dv = (t.cpu() for t in backward(fa.fa_backward_deterministic, qd, kd, vd, o, dod, lse,
                                            wl.scale, wl.causal))
    rows = W.sample_rows(wl.N, 64, seed=9)
    f = parity.f64
    dq_r, dk_r, dv_r = oracle.backward(f(q), f(k), f(v), f(do), wl.scale, causal=wl.causal,
                                       qrows=rows, krows=rows)
    parity.check_grad(dq[:, :, rows], dq_r, "dQ", wl.name)
    parity.check_grad(dk[:, :, rows], dk_r, "dK", wl.name)
    parity.check_grad(dv[:, :, rows], dv_r, "dV", wl.name)
