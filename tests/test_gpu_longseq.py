"""Parity on every long-sequence shape: B*N = 16384 tokens, H = 16,
N in {2048, 4096, 8192, 16384}, d in {64, 128}, causal and not, 1% of the
keys scaled by 8 (the long-range workload and its non-causal twin).  Each
shape runs fa_forward + fa_backward once, in the launch configuration the
benchmark times, and is compared with the fp64 oracle on sampled rows.

Rows: 256 seeded rows plus one seeded row in every 128-row tile, so that
every query tile and every key tile of a checked head is represented (a
wrong tile offset anywhere in a head shows).  The same rows serve as query
rows (O, lse, dQ) and key rows (dK, dV).

Heads: the forward is checked on every (batch, head).  The backward's
oracle needs the full fp64 forward statistics of a head before it can give
any key row's gradient (lse_i and D_i of every query row reaching the
key), about 4 N^2 d flops per head (half when causal).  So the backward is
checked on every head when the shape's heads fit parity.ORACLE_BUDGET
flops, else on a
subset of that size: the first and last head, the first and last head
holding a unit of the persistent backward's last round (on d = 128 dense
shapes those units run as two halves on two CTAs), and seeded others.
"""
import dataclasses

import pytest

from gpu_common import device, status_ok, torch
import parity

import fa_workloads as W
import io_aware_exact_15_gb300 as fa

pytestmark = pytest.mark.gpu

SHAPES = [f"longseq_{kind}_n{N}_d{d}" for kind in ("causal", "dense")
          for d in (64, 128) for N in (2048, 4096, 8192, 16384)]


# Ragged lengths (no multiple of 128) at grids of 1280 two-tile forward CTAs
# and 2560 backward units: the last query and key tiles are partial in
# every head, in the launch forms long sequences take.
RAGGED = [dataclasses.replace(W.WORKLOADS[f"longseq_{kind}_n4096_d{d}"], N=n, B=4,
                              name=f"ragged_{kind}_n{n}_d{d}")
          for kind in ("causal", "dense") for d, n in ((64, 4999), (128, 5000))]


@pytest.mark.parametrize("w", RAGGED, ids=lambda w: w.name)
def test_long_ragged_sequence_parity(w):
    check_long(w)


@pytest.mark.parametrize("name", SHAPES)
def test_long_sequence_parity(name):
    check_long(W.WORKLOADS[name])


def check_long(w):
    dev = device()
    name = w.name
    B, H, N, d = w.B, w.H, w.N, w.d
    q, k, v, do, _ = W.make_inputs(w)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    assert fa.fa_forward(qd, kd, vd, o, lse, B, H, N, d, w.scale, w.causal) == fa.FA_OK
    dq, dk, dv = (torch.full_like(qd, float("nan")) for _ in range(3))
    nbytes = fa.fa_backward_workspace_size(B, H, N, d)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=dev)
    assert fa.fa_backward(qd, kd, vd, o, dod, lse, dq, dk, dv, B, H, N, d, w.scale, w.causal,
                          ws, nbytes) == fa.FA_OK
    status_ok()
    rows = parity.check_rows(N, w.seed + 31)
    ridx = torch.from_numpy(rows)
    o_c, lse_c = o[:, :, ridx].cpu(), lse[:, :, ridx].cpu()
    o_ref, lse_ref = parity.oracle_forward(q, k, v, w.scale, w.causal, rows=rows)
    parity.check_forward(o_c, lse_c, o_ref, lse_ref, f"{name} (all heads)")

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    heads = parity.backward_heads(w, sms)
    dq_r, dk_r, dv_r = parity.oracle_backward(q, k, v, do, w.scale, w.causal, qrows=rows,
                                              krows=rows, heads=heads)
    idx_b = torch.tensor([b for b, _ in heads])
    idx_h = torch.tensor([h for _, h in heads])
    sel = lambda t: t[idx_b, idx_h][:, ridx].cpu()[None]
    what = f"{name} ({len(heads)} of {B * H} heads)"
    parity.check_grad(sel(dq), dq_r, "dQ", what)
    parity.check_grad(sel(dk), dk_r, "dK", what)
    parity.check_grad(sel(dv), dv_r, "dV", what)
