"""Seeded random shapes no parametrized test names: odd batch and head
counts, ragged lengths up to 2600, both head dimensions, dense and causal in turn.
Each runs fa_forward + fa_backward through the C ABI and is compared with
the fp64 oracle on every head: the forward and the gradients on sampled
rows (256 seeded rows and one in every 128-row tile, query and key rows
alike)."""
import dataclasses

import numpy as np
import pytest

from gpu_common import device, status_ok, torch
import parity

import fa_workloads as W
import io_aware_exact_15_gb300 as fa

pytestmark = pytest.mark.gpu


def shapes(n=10, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 4))
        H = int(rng.integers(1, 6))
        N = int(rng.integers(1, 2601))
        d = int(rng.choice([64, 128]))
        causal = i % 2 == 1
        out.append((B, H, N, d, causal, 3000 + i))
    return out


@pytest.mark.parametrize("B,H,N,d,causal,seed", shapes(),
                         ids=lambda x: str(x) if not isinstance(x, bool) else ("causal" if x else "dense"))
def test_random_shape_parity(B, H, N, d, causal, seed):
    dev = device()
    scale = 1.0 / d ** 0.5
    q, k, v, do = W.make_qkv(B, H, N, d, seed=seed)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    assert fa.fa_forward(qd, kd, vd, o, lse, B, H, N, d, scale, causal) == fa.FA_OK
    dq, dk, dv = (torch.full_like(qd, float("nan")) for _ in range(3))
    nbytes = fa.fa_backward_workspace_size(B, H, N, d)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=dev)
    assert fa.fa_backward(qd, kd, vd, o, dod, lse, dq, dk, dv, B, H, N, d, scale, causal,
                          ws, nbytes) == fa.FA_OK
    status_ok()
    what = f"B{B} H{H} N{N} d{d} causal={causal}"
    rows = parity.check_rows(N, seed)
    ridx = torch.from_numpy(rows)
    o_ref, lse_ref = parity.oracle_forward(q, k, v, scale, causal, rows=rows)
    parity.check_forward(o[:, :, ridx].cpu(), lse[:, :, ridx].cpu(), o_ref, lse_ref, what)
    dq_r, dk_r, dv_r = parity.oracle_backward(q, k, v, do, scale, causal, qrows=rows, krows=rows)
    sel = lambda t: t[:, :, ridx].cpu()
    parity.check_grad(sel(dq), dq_r, "dQ", what)
    parity.check_grad(sel(dk), dk_r, "dK", what)
    parity.check_grad(sel(dv), dv_r, "dV", what)
