"""Packed variable-length batches (key-padding mask as sequence lengths):
q [H, total, d], k/v [Hkv, total, d], sequence b in rows
cu_seqlens[b] .. cu_seqlens[b+1].  CUDA path vs the fp64 oracle's
per-sequence evaluation, forward and backward, with ragged tails, empty
sequences, single-row sequences and grouped heads; plus a bit-exact check
that a packed batch gives each sequence what a call on that sequence alone
gives (O, lse, dK, dV)."""
import numpy as np
import pytest

from gpu_common import device, status_ok, torch
import parity

import fa_workloads as W
import io_aware_exact_15_gb300 as fa
import oracle

pytestmark = pytest.mark.gpu


def make(H, Hkv, lens, d, seed):
    g = torch.Generator().manual_seed(seed)
    T = int(sum(lens))
    q = W.randn_bf16((H, T, d), g)
    k = W.randn_bf16((Hkv, T, d), g)
    v = W.randn_bf16((Hkv, T, d), g)
    do = W.randn_bf16((H, T, d), g)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return q, k, v, do, cu


def run(q, k, v, do, cu, scale, causal, dev, backward=True, drop=(0.0, 0, 0)):
    H, T, d = q.shape
    Hkv = k.shape[0]
    B = len(cu) - 1
    ms = int(np.max(np.diff(cu))) if T > 0 else 0
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    cud = torch.from_numpy(cu).to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((H, T), float("nan"), dtype=torch.float32, device=dev)
    assert fa.fa_forward_varlen(qd, kd, vd, o, lse, cud, B, ms, T, H, Hkv, d, scale,
                                causal, *drop) == fa.FA_OK
    out = [o, lse]
    if backward:
        dq = torch.full_like(qd, float("nan"))
        dk, dv = torch.full_like(kd, float("nan")), torch.full_like(vd, float("nan"))
        nbytes = fa.fa_backward_workspace_size(1, H, T, d)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        assert fa.fa_backward_varlen(qd, kd, vd, o, dod, lse, dq, dk, dv, cud, B, ms, T, H, Hkv, d,
                                     scale, causal, *drop, ws, nbytes) == fa.FA_OK
        out += [dq, dk, dv]
    status_ok()
    return [t.cpu() for t in out]


LENS = {
    "ragged": [200, 1, 0, 383, 128, 77],
    "tiles": [256, 128, 129, 255],
    "one_long": [700, 3],
    "single": [300],
}


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hkv", [(4, 4), (6, 2)])
@pytest.mark.parametrize("mix", sorted(LENS))
def test_varlen_small_full(mix, H, Hkv, d, causal):
    dev = device()
    lens = LENS[mix]
    q, k, v, do, cu = make(H, Hkv, lens, d, seed=sum(lens) + 10 * H + Hkv + d + causal)
    scale = 1.0 / d ** 0.5
    o, lse, dq, dk, dv = run(q, k, v, do, cu, scale, causal, dev)
    what = f"{mix} H={H} Hkv={Hkv} d={d} causal={causal}"
    f = parity.f64
    o_ref, lse_ref = oracle.forward_varlen(f(q), f(k), f(v), cu, scale, causal=causal)
    parity.check_forward(o, lse, o_ref, lse_ref, what)
    dq_r, dk_r, dv_r = oracle.backward_varlen(f(q), f(k), f(v), f(do), cu, scale, causal=causal)
    parity.check_grad(dq, dq_r, "dQ", what)
    parity.check_grad(dk, dk_r, "dK", what)
    parity.check_grad(dv, dv_r, "dV", what)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_separate_calls(causal):
    """Each sequence of a packed batch gets exactly the O, lse, dK, dV of a
    B = 1 call on that sequence alone (dQ is summed by unordered atomic adds,
    so it is compared within tolerance instead)."""
    dev = device()
    lens = [333, 128, 1, 512, 90]
    H, d = 4, 64
    q, k, v, do, cu = make(H, H, lens, d, seed=31 + causal)
    scale = 0.125
    o, lse, dq, dk, dv = run(q, k, v, do, cu, scale, causal, dev)
    for a, b in zip(cu[:-1], cu[1:]):
        n = int(b - a)
        qs, ks, vs, dos = (t[None, :, a:b].contiguous().to(dev) for t in (q, k, v, do))
        os_ = torch.empty_like(qs)
        ls = torch.empty((1, H, n), dtype=torch.float32, device=dev)
        assert fa.fa_forward(qs, ks, vs, os_, ls, 1, H, n, d, scale, causal) == fa.FA_OK
        dqs, dks, dvs = torch.empty_like(qs), torch.empty_like(ks), torch.empty_like(vs)
        nbytes = fa.fa_backward_workspace_size(1, H, n, d)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        assert fa.fa_backward(qs, ks, vs, os_, dos, ls, dqs, dks, dvs, 1, H, n, d, scale, causal,
                              ws, nbytes) == fa.FA_OK
        status_ok()
        assert torch.equal(o[:, a:b], os_[0].cpu()), (a, b)
        assert torch.equal(lse[:, a:b], ls[0].cpu()), (a, b)
        assert torch.equal(dk[:, a:b], dks[0].cpu()), (a, b)
        assert torch.equal(dv[:, a:b], dvs[0].cpu()), (a, b)
        parity.check_grad(dq[:, a:b], parity.f64(dqs[0]), "dQ", f"seq {a}:{b}")


def test_varlen_all_empty_and_empty_edges():
    dev = device()
    H, d = 2, 64
    # every sequence empty: nothing to do, FA_OK, nothing launched (an
    # aligned dummy buffer stands in for the empty tensors)
    buf = torch.zeros(1024, dtype=torch.bfloat16, device=dev)
    cu = torch.zeros(4, dtype=torch.int32, device=dev)
    assert fa.fa_forward_varlen(buf, buf, buf, buf, buf, cu, 3, 0, 0, H, H, d, 0.125, 0, 0.0, 0,
                                0) == fa.FA_OK
    assert fa.fa_backward_varlen(buf, buf, buf, buf, buf, buf, buf, buf, buf, cu, 3, 0, 0, H, H,
                                 d, 0.125, 0, 0.0, 0, 0, buf, buf.numel() * 2) == fa.FA_OK
    status_ok()
    assert not buf.any()
    # empty sequences first and last around a ragged one
    q, k, v, do, cun = make(H, H, [0, 0, 150, 0], d, seed=5)
    o, lse2, dq, dk, dv = run(q, k, v, do, cun, 0.125, True, dev)
    f = parity.f64
    o_ref, lse_ref = oracle.forward_varlen(f(q), f(k), f(v), cun, 0.125, causal=True)
    parity.check_forward(o, lse2, o_ref, lse_ref, "empty edges")
    dq_r, dk_r, dv_r = oracle.backward_varlen(f(q), f(k), f(v), f(do), cun, 0.125, causal=True)
    parity.check_grad(dq, dq_r, "dQ", "empty edges")
    parity.check_grad(dk, dk_r, "dK", "empty edges")
    parity.check_grad(dv, dv_r, "dV", "empty edges")


def test_varlen_workload_sampled_rows():
    """The packed BERT-large-shaped batch (8 sequences of 128..512 rows,
    16 heads, d = 64) as the benchmark runs it; oracle on sampled rows of
    every sequence."""
    dev = device()
    wl = W.WORKLOADS["bert_large_varlen"]
    q, k, v, do, cu = W.make_varlen_inputs(wl)
    scale = wl.scale
    o, lse, dq, dk, dv = run(q, k, v, do, cu, scale, wl.causal, dev)
    f = parity.f64
    for i, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        n = int(b - a)
        rows = W.sample_rows(n, 24, seed=i)
        sl = slice(int(a), int(b))
        qs, ks, vs, dos = (f(t[None, :, sl]) for t in (q, k, v, do))
        o_ref, lse_ref = oracle.forward(qs, ks, vs, scale, causal=wl.causal, rows=rows)
        parity.check_forward(o[None, :, sl][:, :, rows], lse[None, :, sl][:, :, rows], o_ref,
                             lse_ref, f"seq {i}")
        dq_r, dk_r, dv_r = oracle.backward(qs, ks, vs, dos, scale, causal=wl.causal, qrows=rows,
                                           krows=rows)
        parity.check_grad(dq[None, :, sl][:, :, rows], dq_r, "dQ", f"seq {i}")
        parity.check_grad(dk[None, :, sl][:, :, rows], dk_r, "dK", f"seq {i}")
        parity.check_grad(dv[None, :, sl][:, :, rows], dv_r, "dV", f"seq {i}")


@pytest.mark.parametrize("p_drop", [0.0, 0.2])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_varlen_large_batch_two_tile_path(d, causal, p_drop):
    # Ten sequences up to 1100 tokens with 16 query heads over 4 K/V heads:
    # 5 query-tile pairs x 10 x 16 = 800 CTAs of two tiles, more than the
    # forward's small-grid limit (4 x 152), so the two-tile form runs here
    # (the small batches above take the compact one-tile form).
    dev = device()
    rng = np.random.default_rng(77 + d + causal)
    lens = [1100, 0, 1] + [int(x) for x in rng.integers(200, 1101, 7)]
    H, Hkv = 16, 4
    q, k, v, do, cu = make(H, Hkv, lens, d, seed=sum(lens) + d + causal)
    scale = 1.0 / d ** 0.5
    drop = (p_drop, 0x5EED + d, 11) if p_drop > 0 else (0.0, 0, 0)
    o, lse, dq, dk, dv = run(q, k, v, do, cu, scale, causal, dev, drop=drop)
    what = f"large varlen d={d} causal={causal} p={p_drop}"
    f = parity.f64
    od = drop if p_drop > 0 else None
    o_ref, lse_ref = oracle.forward_varlen(f(q), f(k), f(v), cu, scale, causal=causal, dropout=od)
    parity.check_forward(o, lse, o_ref, lse_ref, what, o_scale=parity.keep_scale(p_drop))
    dq_r, dk_r, dv_r = oracle.backward_varlen(f(q), f(k), f(v), f(do), cu, scale, causal=causal,
                                              dropout=od)
    parity.check_grad(dq, dq_r, "dQ", what)
    parity.check_grad(dk, dk_r, "dK", what)
    parity.check_grad(dv, dv_r, "dV", what)
