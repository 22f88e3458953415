"""The persistent backward under load: shapes with more key-tile units than
SMs (so every CTA walks several units and crosses unit boundaries), each run
several times.  dK and dV must equal the deterministic key-tile pass bit for
bit (same products in the same order; to tolerance where the last round is
split into halves), dQ must agree with the deterministic dQ pass within the
gradient tolerance, and repeated runs must give the same dK, dV and (to
rounding) dQ: a missing or doubled reduce-add, or a staging buffer
overwritten before the TMA read it, shows up as a whole key tile's
contribution to one slice of dQ."""
import pytest

from gpu_common import device, status_ok, torch
import parity

import fa_workloads as W
import io_aware_exact_15_gb300 as fa

pytestmark = pytest.mark.gpu

RUNS = 3


def _forward(qd, kd, vd, scale, causal):
    B, H, N, d = qd.shape
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=qd.device)
    assert fa.fa_forward(qd, kd, vd, o, lse, B, H, N, d, scale, causal) == fa.FA_OK
    return o, lse


def _backward(fn, qd, kd, vd, o, dod, lse, scale, causal):
    B, H, N, d = qd.shape
    dq, dk, dv = (torch.full_like(qd, float("nan")) for _ in range(3))
    nbytes = fa.fa_backward_workspace_size(B, H, N, d)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=qd.device)
    assert fn(qd, kd, vd, o, dod, lse, dq, dk, dv, B, H, N, d, scale, causal, ws,
              nbytes) == fa.FA_OK
    status_ok()
    return dq, dk, dv


def _splits(B, H, N, d, causal):
    """Whether the persistent backward splits its last round: one CTA per
    SM; the d = 128 kernel splits the last round when it holds at most half
    the grid, fits the workspace's slots (units / 2, at most 96) and its
    units have at least 8 steps (nT dense, 1 causal, with one query head per
    key/value head)."""
    if d != 128:
        return False
    nT = (N + 127) // 128
    units = B * H * nT
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    grid = min(units, sms)
    rounds = (units + grid - 1) // grid
    mlast = units - (rounds - 1) * grid
    slots = min(units // 2, 96) if units > 64 else 0
    return (rounds > 1 and 2 * mlast <= grid and mlast <= slots and
            (1 if causal else nT) >= 8)


# (B, H, N, d): 160 to 1024 key-tile units for the 152-SM grid.  Where the
# last round holds at most half the grid and its units are long enough (d =
# 128, 160 and 192 units, dense: 8 and 40 units of 10 and 12 steps left
# over) those units run as two halves on two CTAs, whose dK, dV partial sums
# meet in the workspace.
SHAPES = [(2, 8, 2048, 128), (4, 16, 512, 64), (2, 16, 1024, 64), (1, 8, 4096, 128),
          (2, 8, 1280, 128), (1, 16, 1536, 128)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", SHAPES)
def test_multi_unit_backward_consistent(B, H, N, d, causal):
    dev = device()
    q, k, v, do = W.make_qkv(B, H, N, d, seed=900 + N + d + B + causal)
    scale = 1.0 / d ** 0.5
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = _forward(qd, kd, vd, scale, causal)
    dq_det, dk_det, dv_det = _backward(fa.fa_backward_deterministic, qd, kd, vd, o, dod, lse,
                                       scale, causal)
    ref = parity.f64(dq_det.cpu())
    what = f"B{B} H{H} N{N} d{d} causal={causal}"
    split = _splits(B, H, N, d, causal)
    first = None
    for run in range(RUNS):
        dq, dk, dv = _backward(fa.fa_backward, qd, kd, vd, o, dod, lse, scale, causal)
        if split:
            # a split unit's dK, dV is the sum of its two halves' partial
            # sums (another fp32 order than one pass): equal to tolerance
            parity.check_grad(dk.cpu(), parity.f64(dk_det.cpu()), "dK", what)
            parity.check_grad(dv.cpu(), parity.f64(dv_det.cpu()), "dV", what)
        else:
            assert torch.equal(dk, dk_det), f"{what} run {run}: dK differs from the key-tile pass"
            assert torch.equal(dv, dv_det), f"{what} run {run}: dV differs from the key-tile pass"
        parity.check_grad(dq.cpu(), ref, "dQ", f"{what} run {run} vs deterministic dQ")
        if first is None:
            first = (dq, dk, dv)
        else:
            # dK, dV: the same sums every run (own half + parked half, which
            # commute exactly); dQ: reduce-adds commute only to rounding
            assert torch.equal(dk, first[1]) and torch.equal(dv, first[2]), \
                f"{what} run {run}: dK/dV changed between runs"
            assert (dq.float() - first[0].float()).abs().max().item() <= \
                1e-2 * first[0].float().abs().max().item(), f"{what} run {run}: dQ drifted"


@pytest.mark.parametrize("B,H,N,d", [(2, 8, 1280, 128), (1, 16, 1536, 128), (2, 8, 5000, 128)])
def test_split_last_round_against_oracle(B, H, N, d):
    # The last round's units run as two halves whose dK, dV partial sums
    # meet in the workspace.  Every row of every head that holds a
    # last-round unit is compared with the fp64 oracle: B2 H8 N1280 leaves
    # units 152..159 (head 15, key tiles 2..9), B1 H16 N1536 units 152..191
    # (heads 12..15) on the 152-SM grid; B2 H8 N5000 units 608..639 (head
    # 15), whose halves walk 40 query tiles, the last one partial.
    dev = device()
    assert _splits(B, H, N, d, False), "shape no longer splits its last round"
    q, k, v, do = W.make_qkv(B, H, N, d, seed=4100 + N + B)
    scale = 1.0 / d ** 0.5
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = _forward(qd, kd, vd, scale, False)
    dq, dk, dv = _backward(fa.fa_backward, qd, kd, vd, o, dod, lse, scale, False)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    heads = parity.last_round_heads(B, H, N, False, sms)
    dq_r, dk_r, dv_r = parity.oracle_backward(q, k, v, do, scale, False, heads=heads)
    sel = lambda t: torch.stack([t[b, h] for (b, h) in heads]).cpu()[None]
    what = f"B{B} H{H} N{N} d{d} last-round heads {heads}"
    parity.check_grad(sel(dk), dk_r, "dK", what)
    parity.check_grad(sel(dv), dv_r, "dV", what)
    parity.check_grad(sel(dq), dq_r, "dQ", what)
