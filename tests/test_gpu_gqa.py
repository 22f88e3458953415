"""Grouped key/value heads: H query heads over Hkv K/V heads (Hkv = 1 is
multi-query attention).  CUDA path vs the fp64 oracle, forward and backward;
dK/dV are the sums over each group's query heads."""
import numpy as np
import pytest

from gpu_common import device, status_ok, torch
import parity

import fa_workloads as W
import io_aware_exact_15_gb300 as fa
import oracle

pytestmark = pytest.mark.gpu


def make(B, H, Hkv, N, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = W.randn_bf16((B, H, N, d), g)
    k = W.randn_bf16((B, Hkv, N, d), g)
    v = W.randn_bf16((B, Hkv, N, d), g)
    do = W.randn_bf16((B, H, N, d), g)
    return q, k, v, do


def run(q, k, v, do, scale, causal, dev):
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    assert fa.fa_forward_gqa(qd, kd, vd, o, lse, B, H, Hkv, N, d, scale, causal) == fa.FA_OK
    dq = torch.full_like(qd, float("nan"))
    dk, dv = torch.full_like(kd, float("nan")), torch.full_like(vd, float("nan"))
    nbytes = fa.fa_backward_workspace_size(B, H, N, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    assert fa.fa_backward_gqa(qd, kd, vd, o, dod, lse, dq, dk, dv, B, H, Hkv, N, d, scale, causal,
                              ws, nbytes) == fa.FA_OK
    status_ok()
    return [t.cpu() for t in (o, lse, dq, dk, dv)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hkv,N", [(6, 1, 200), (6, 2, 384), (4, 4, 257), (8, 2, 130)])
def test_gqa_small_full(H, Hkv, N, d, causal):
    dev = device()
    q, k, v, do = make(2, H, Hkv, N, d, seed=H * 100 + Hkv * 10 + N + d + causal)
    scale = 1.0 / d ** 0.5
    o, lse, dq, dk, dv = run(q, k, v, do, scale, causal, dev)
    what = f"H={H} Hkv={Hkv} N={N} d={d} causal={causal}"
    f = parity.f64
    o_ref, lse_ref = oracle.forward(f(q), f(k), f(v), scale, causal=causal)
    parity.check_forward(o, lse, o_ref, lse_ref, what)
    dq_r, dk_r, dv_r = oracle.backward(f(q), f(k), f(v), f(do), scale, causal=causal)
    parity.check_grad(dq, dq_r, "dQ", what)
    parity.check_grad(dk, dk_r, "dK", what)
    parity.check_grad(dv, dv_r, "dV", what)


def test_gqa_equals_mha_when_groups_are_single():
    dev = device()
    q, k, v, do = make(1, 4, 4, 300, 64, seed=8)
    a = run(q, k, v, do, 0.125, True, dev)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((1, 4, 300), dtype=torch.float32, device=dev)
    assert fa.fa_forward(qd, kd, vd, o, lse, 1, 4, 300, 64, 0.125, 1) == fa.FA_OK
    status_ok()
    assert torch.equal(a[0], o.cpu()) and torch.equal(a[1], lse.cpu())


def test_gqa_long_sequence_sampled_rows():
    dev = device()
    B, H, Hkv, N, d = 2, 16, 4, 2048, 128
    q, k, v, do = make(B, H, Hkv, N, d, seed=2024)
    scale = 1.0 / d ** 0.5
    o, lse, dq, dk, dv = run(q, k, v, do, scale, True, dev)
    rows = W.sample_rows(N, 256, seed=77)
    f = parity.f64
    o_ref, lse_ref = oracle.forward(f(q), f(k), f(v), scale, causal=True, rows=rows)
    parity.check_forward(o[:, :, rows], lse[:, :, rows], o_ref, lse_ref, "gqa 2k")
    dq_r, dk_r, dv_r = oracle.backward(f(q), f(k), f(v), f(do), scale, causal=True, qrows=rows,
                                       krows=rows)
    parity.check_grad(dq[:, :, rows], dq_r, "dQ", "gqa 2k")
    parity.check_grad(dk[:, :, rows], dk_r, "dK", "gqa 2k")
    parity.check_grad(dv[:, :, rows], dv_r, "dV", "gqa 2k")


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_split_last_round_sampled_rows(causal):
    # 2 x 4 key/value heads x 20 key tiles = 160 units on the 152-SM grid:
    # dense, the 8 units of the last round (4 x 20 steps each) run as two
    # halves each (the d = 128 kernel; d = 64 never splits); causal ones
    # (4 steps) do not split.  The key rows checked
    # include every row of the key tiles those units own
    dev = device()
    B, H, Hkv, N, d = 2, 16, 4, 2560, 128
    q, k, v, do = make(B, H, Hkv, N, d, seed=31 + causal)
    scale = 1.0 / d ** 0.5
    o, lse, dq, dk, dv = run(q, k, v, do, scale, causal, dev)
    # last-round units: causal walks key tile 19 of every head first-to-last
    # (units 152..159 are (kt 19, heads 0..7)); dense ones are key tiles 12..19
    # of the last key/value head
    last = list(range(19 * 128, 20 * 128)) if causal else list(range(12 * 128, 13 * 128))
    krows = np.unique(np.concatenate([np.array(last), W.sample_rows(N, 64, seed=5)]))
    qrows = W.sample_rows(N, 64, seed=6)
    f = parity.f64
    dq_r, dk_r, dv_r = oracle.backward(f(q), f(k), f(v), f(do), scale, causal=causal, qrows=qrows,
                                       krows=krows)
    what = f"gqa split causal={causal}"
    parity.check_grad(dq[:, :, qrows], dq_r, "dQ", what)
    parity.check_grad(dk[:, :, krows], dk_r, "dK", what)
    parity.check_grad(dv[:, :, krows], dv_r, "dV", what)


def test_gqa_causal_split_last_round_eight_heads_per_group():
    # 4 x 2 key/value heads x 20 key tiles = 160 units, causal, 8 query heads
    # per key/value head: the last round holds the 8 diagonal units of key
    # tile 19, 8 steps each (one per query head), which run as two halves of
    # 4 steps on two CTAs.  Every row of key tile 19 is checked.
    dev = device()
    B, H, Hkv, N, d = 4, 16, 2, 2560, 128
    q, k, v, do = make(B, H, Hkv, N, d, seed=77)
    scale = 1.0 / d ** 0.5
    o, lse, dq, dk, dv = run(q, k, v, do, scale, True, dev)
    krows = np.unique(np.concatenate([np.arange(19 * 128, 20 * 128), W.sample_rows(N, 32, seed=8)]))
    qrows = W.sample_rows(N, 48, seed=9)
    f = parity.f64
    dq_r, dk_r, dv_r = oracle.backward(f(q), f(k), f(v), f(do), scale, causal=True, qrows=qrows,
                                       krows=krows)
    what = "gqa causal split, 8 heads per group"
    parity.check_grad(dq[:, :, qrows], dq_r, "dQ", what)
    parity.check_grad(dk[:, :, krows], dk_r, "dK", what)
    parity.check_grad(dv[:, :, krows], dv_r, "dV", what)
