"""Dropout on P fused into both passes: CUDA path vs the fp64 oracle with the
same Philox keep rule, and a bit-exact read-out of the forward kernel's
keep decisions."""
import numpy as np
import pytest

from gpu_common import device, status_ok, torch
import parity

import fa_workloads as W
import io_aware_exact_15_gb300 as fa
import oracle

pytestmark = pytest.mark.gpu


def run(q, k, v, do, scale, causal, drop, dev):
    B, H, N, d = q.shape
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    assert fa.fa_forward_dropout(qd, kd, vd, o, lse, B, H, N, d, scale, causal, *drop) == fa.FA_OK
    dq, dk, dv = (torch.full_like(qd, float("nan")) for _ in range(3))
    nbytes = fa.fa_backward_workspace_size(B, H, N, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    assert fa.fa_backward_dropout(qd, kd, vd, o, dod, lse, dq, dk, dv, B, H, N, d, scale, causal,
                                  *drop, ws, nbytes) == fa.FA_OK
    status_ok()
    return [t.cpu() for t in (o, lse, dq, dk, dv)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,p", [(200, 0.1), (384, 0.5), (1, 0.3), (257, 0.9)])
def test_dropout_small_full(N, p, d, causal):
    dev = device()
    q, k, v, do = W.make_qkv(2, 3, N, d, seed=N + d + causal + int(p * 100))
    scale = 1.0 / d ** 0.5
    drop = (p, 0x1234_5678_9ABC + N, 7 + d)
    o, lse, dq, dk, dv = run(q, k, v, do, scale, causal, drop, dev)
    what = f"N={N} d={d} p={p} causal={causal}"
    f = parity.f64
    o_ref, lse_ref = oracle.forward(f(q), f(k), f(v), scale, causal=causal, dropout=drop)
    parity.check_forward(o, lse, o_ref, lse_ref, what, o_scale=parity.keep_scale(p))
    dq_r, dk_r, dv_r = oracle.backward(f(q), f(k), f(v), f(do), scale, causal=causal,
                                       dropout=drop)
    # N = 1: dQ = dK = 0 exactly by cancellation; bound by the cancelling
    # terms' scale (D comes from the bf16-rounded O = z v / (1 - p')), taken
    # from the oracle's O rounded to bf16, never from the output under test
    o_b = torch.from_numpy(o_ref).to(torch.bfloat16)
    fq = parity.cancel_floor(scale, o_b, do, k) if N == 1 else parity.GRAD_FLOOR
    fk = parity.cancel_floor(scale, o_b, do, q) if N == 1 else parity.GRAD_FLOOR
    parity.check_grad(dq, dq_r, "dQ", what, floor=fq)
    parity.check_grad(dk, dk_r, "dK", what, floor=fk)
    parity.check_grad(dv, dv_r, "dV", what)


@pytest.mark.parametrize("d,H", [(64, 2), (128, 2), (64, 320), (128, 160)])
def test_forward_keep_bits_are_exact(d, H):
    """Q = 0 makes every weight 1 before normalisation, p = 1/2 makes the
    keep scale 2, and V puts weight 2^(j // d) on column j mod d of key j,
    so with N = 8 d every intermediate is exact and O_ic * N / 2 is the
    8-bit number whose bit t is the keep decision of key t d + c.  That
    reads out the kernel's decision for every (row, key), to be equal to
    the oracle's keep rule.  H = 2 runs the compact one-tile form (the
    softmax warps draw the bits); 320 and 160 heads make grids of 640
    two-tile CTAs, where two warps of their own draw them."""
    dev = device()
    B, N = 1, 8 * d
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16)
    g = torch.Generator().manual_seed(3)
    k = W.randn_bf16((B, H, N, d), g)
    j = np.arange(N)
    vv = np.zeros((N, d), dtype=np.float32)
    vv[j, j % d] = 2.0 ** (j // d)
    v = torch.from_numpy(vv).to(torch.bfloat16).expand(B, H, N, d).contiguous()
    seed, offset = 0xDEADBEEF_0BADF00D, 12345
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    assert fa.fa_forward_dropout(qd, kd, vd, o, lse, B, H, N, d, 1.0, 0, 0.5, seed,
                                 offset) == fa.FA_OK
    status_ok()
    code = o.float().cpu().numpy() * (N / 2)
    assert np.array_equal(code, np.rint(code)), "O is not an exact multiple of 2/N"
    code = code.astype(np.uint8)                                   # [B, H, N, d]
    bits = (code[..., None] >> np.arange(8, dtype=np.uint8)) & 1   # [B, H, N, d, 8]
    z_gpu = bits.transpose(0, 1, 2, 4, 3).reshape(B, H, N, N)      # key = t d + c
    z_ref = oracle.dropout_keep(seed, offset, 0.5, B, H, N)
    assert np.array_equal(z_gpu, z_ref), f"{int((z_gpu != z_ref).sum())} keep bits differ"


def test_p_zero_is_the_plain_path():
    dev = device()
    q, k, v, do = W.make_qkv(1, 2, 300, 64, seed=5)
    a = run(q, k, v, do, 0.125, True, (0.0, 99, 1), dev)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((1, 2, 300), dtype=torch.float32, device=dev)
    assert fa.fa_forward(qd, kd, vd, o, lse, 1, 2, 300, 64, 0.125, 1) == fa.FA_OK
    status_ok()
    assert torch.equal(a[0], o.cpu()) and torch.equal(a[1], lse.cpu())


def test_offset_and_seed_change_the_mask():
    """A different offset or seed draws a different mask: the outputs move
    by about the dropout noise, while lse (undropped) stays bit-identical."""
    dev = device()
    q, k, v, do = W.make_qkv(1, 2, 256, 64, seed=6)
    outs = [run(q, k, v, do, 0.125, False, drop, dev)
            for drop in ((0.2, 1, 0), (0.2, 1, 1), (0.2, 2, 0), (0.2, 1, 0))]
    assert torch.equal(outs[0][0], outs[3][0])        # same (seed, offset): same O
    for other in outs[1:3]:
        assert not torch.equal(outs[0][0], other[0])
        assert torch.equal(outs[0][1], other[1])


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_dropout_small(causal):
    dev = device()
    lens = [200, 0, 1, 383, 128]
    H, d = 4, 64
    g = torch.Generator().manual_seed(50 + causal)
    T = sum(lens)
    q, k, v, do = (W.randn_bf16((H, T, d), g) for _ in range(4))
    cu = W.cu_seqlens(lens)
    drop = (0.15, 77, 3)
    cud = torch.from_numpy(cu).to(dev)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    B, ms = len(lens), max(lens)
    assert fa.fa_forward_varlen(qd, kd, vd, o, lse, cud, B, ms, T, H, H, d, 0.125, causal,
                                *drop) == fa.FA_OK
    dq, dk, dv = (torch.empty_like(qd) for _ in range(3))
    nbytes = fa.fa_backward_workspace_size(1, H, T, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    assert fa.fa_backward_varlen(qd, kd, vd, o, dod, lse, dq, dk, dv, cud, B, ms, T, H, H, d,
                                 0.125, causal, *drop, ws, nbytes) == fa.FA_OK
    status_ok()
    f = parity.f64
    o_ref, lse_ref = oracle.forward_varlen(f(q), f(k), f(v), cu, 0.125, causal=causal,
                                           dropout=drop)
    parity.check_forward(o.cpu(), lse.cpu(), o_ref, lse_ref, "varlen dropout",
                         o_scale=parity.keep_scale(drop[0]))
    g_ref = oracle.backward_varlen(f(q), f(k), f(v), f(do), cu, 0.125, causal=causal,
                                   dropout=drop)
    for name, a, b in zip(("dQ", "dK", "dV"), (dq, dk, dv), g_ref):
        parity.check_grad(a.cpu(), b, name, "varlen dropout")


def test_longseq_dropout_sampled_rows():
    """longseq_dense_n4096_d128_dropout as the benchmark runs it; the oracle
    on 64 sampled rows of every head."""
    dev = device()
    wl = W.WORKLOADS["longseq_dense_n4096_d128_dropout"]
    q, k, v, do, _ = W.make_inputs(wl)
    drop = (wl.dropout, W.DROPOUT_SEED, 0)
    o, lse, dq, dk, dv = run(q, k, v, do, wl.scale, wl.causal, drop, dev)
    rows = W.sample_rows(wl.N, 64, seed=123)
    f = parity.f64
    o_ref, lse_ref = oracle.forward(f(q), f(k), f(v), wl.scale, causal=wl.causal, rows=rows,
                                    dropout=drop)
    parity.check_forward(o[:, :, rows], lse[:, :, rows], o_ref, lse_ref, wl.name,
                         o_scale=parity.keep_scale(wl.dropout))
    dq_r, dk_r, dv_r = oracle.backward(f(q), f(k), f(v), f(do), wl.scale, causal=wl.causal,
                                       qrows=rows, krows=rows, dropout=drop)
    parity.check_grad(dq[:, :, rows], dq_r, "dQ", wl.name)
    parity.check_grad(dk[:, :, rows], dk_r, "dK", wl.name)
    parity.check_grad(dv[:, :, rows], dv_r, "dV", wl.name)


def test_varlen_dropout_workload_sampled_rows():
    dev = device()
    wl = W.WORKLOADS["bert_large_varlen_dropout"]
    q, k, v, do, cu = W.make_varlen_inputs(wl)
    drop = (wl.dropout, W.DROPOUT_SEED, 0)
    H, T, d = q.shape
    cud = torch.from_numpy(cu).to(dev)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    B, ms = len(cu) - 1, int(np.diff(cu).max())
    assert fa.fa_forward_varlen(qd, kd, vd, o, lse, cud, B, ms, T, H, H, d, wl.scale, wl.causal,
                                *drop) == fa.FA_OK
    dq, dk, dv = (torch.empty_like(qd) for _ in range(3))
    nbytes = fa.fa_backward_workspace_size(1, H, T, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    assert fa.fa_backward_varlen(qd, kd, vd, o, dod, lse, dq, dk, dv, cud, B, ms, T, H, H, d,
                                 wl.scale, wl.causal, *drop, ws, nbytes) == fa.FA_OK
    status_ok()
    o, lse, dq, dk, dv = (t.cpu() for t in (o, lse, dq, dk, dv))
    f = parity.f64
    for i, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        rows = W.sample_rows(int(b - a), 24, seed=i)
        sl = slice(int(a), int(b))
        qs, ks, vs, dos = (f(t[None, :, sl]) for t in (q, k, v, do))
        o_ref, lse_ref = oracle.forward(qs, ks, vs, wl.scale, causal=wl.causal, rows=rows,
                                        dropout=drop, batch0=i)
        parity.check_forward(o[None, :, sl][:, :, rows], lse[None, :, sl][:, :, rows], o_ref,
                             lse_ref, f"seq {i}", o_scale=parity.keep_scale(wl.dropout))
        g_ref = oracle.backward(qs, ks, vs, dos, wl.scale, causal=wl.causal, qrows=rows,
                                krows=rows, dropout=drop, batch0=i)
        for name, a_, b_ in zip(("dQ", "dK", "dV"), (dq, dk, dv), g_ref):
            parity.check_grad(a_[None, :, sl][:, :, rows], b_, name, f"seq {i}")
