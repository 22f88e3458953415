"""Block-sparse parity and the bit-exact integer work (tile lists, schedules)."""
import numpy as np
import pytest

from gpu_common import device, status_ok, torch
import parity

import fa_workloads as W
import io_aware_exact_15_gb300 as fa
import oracle

pytestmark = pytest.mark.gpu


def run_sparse(q, k, v, do, scale, causal, mask, dev):
    B, H, N, d = q.shape
    mh = mask.shape[0]
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = torch.from_numpy(np.ascontiguousarray(mask)).to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    nbytes = fa.fa_blocksparse_workspace_size(B, H, N, d, mh)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    assert fa.fa_blocksparse_forward(qd, kd, vd, o, lse, B, H, N, d, scale, causal, md, mh, ws,
                                     nbytes) == fa.FA_OK
    out = [o, lse]
    if do is not None:
        dod = do.to(dev)
        dq, dk, dv = (torch.full_like(qd, float("nan")) for _ in range(3))
        assert fa.fa_blocksparse_backward(qd, kd, vd, o, dod, lse, dq, dk, dv, B, H, N, d, scale,
                                          causal, md, mh, ws, nbytes) == fa.FA_OK
        out += [dq, dk, dv]
    status_ok()
    return [t.cpu() for t in out]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,mh", [(300, 1), (640, 2), (1000, 1)])
def test_blocksparse_small_full(N, mh, d, causal):
    dev = device()
    B, H = 1, 2
    nT = (N + 127) // 128
    q, k, v, do = W.make_qkv(B, H, N, d, seed=N + d + causal)
    mask = W.random_block_mask(mh, nT, seed=N + 1, density=0.45)
    mask[0, 1, :] = 0  # a query tile with no kept key tile
    mask[-1, :, 0] = 1
    scale = 1.0 / d ** 0.5
    o, lse, dq, dk, dv = run_sparse(q, k, v, do, scale, causal, mask, dev)
    what = f"N={N} mh={mh} d={d} causal={causal}"
    o_ref, lse_ref = parity.oracle_forward(q, k, v, scale, causal, mask=mask)
    parity.check_forward(o, lse, o_ref, lse_ref, what)
    dq_r, dk_r, dv_r = parity.oracle_backward(q, k, v, do, scale, causal, mask=mask)
    parity.check_grad(dq, dq_r, "dQ", what)
    parity.check_grad(dk, dk_r, "dK", what)
    parity.check_grad(dv, dv_r, "dV", what)


def test_blocksparse_all_ones_equals_dense():
    dev = device()
    q, k, v, _ = W.make_qkv(1, 2, 384, 64, seed=9, with_do=False)
    mask = np.ones((1, 3, 3), dtype=np.uint8)
    o_s, lse_s = run_sparse(q, k, v, None, 0.125, False, mask, dev)
    o_d = torch.empty_like(q.to(dev))
    lse_d = torch.empty((1, 2, 384), dtype=torch.float32, device=dev)
    assert fa.fa_forward(q.to(dev), k.to(dev), v.to(dev), o_d, lse_d, 1, 2, 384, 64, 0.125,
                         0) == fa.FA_OK
    status_ok()
    assert torch.equal(o_s, o_d.cpu()) and torch.equal(lse_s, lse_d.cpu())


def test_blocksparse_64k_sampled_rows():
    # every head, 256 seeded rows plus one row in each of the 512 tiles (the
    # oracle's per-head cost is the sparse forward statistics, ~5.7 % of
    # the dense 4 N^2 d)
    dev = device()
    w = W.WORKLOADS["blocksparse_64k"]
    q, k, v, do, mask = W.make_inputs(w)
    o, lse, dq, dk, dv = run_sparse(q, k, v, do, w.scale, w.causal, mask, dev)
    rows = parity.check_rows(w.N, seed=w.seed + 29)
    o_ref, lse_ref = parity.oracle_forward(q, k, v, w.scale, w.causal, mask=mask, rows=rows)
    parity.check_forward(o[:, :, rows], lse[:, :, rows], o_ref, lse_ref, "blocksparse_64k")
    dq_r, dk_r, dv_r = parity.oracle_backward(q, k, v, do, w.scale, w.causal, mask=mask,
                                              qrows=rows, krows=rows)
    parity.check_grad(dq[:, :, rows], dq_r, "dQ", "blocksparse_64k")
    parity.check_grad(dk[:, :, rows], dk_r, "dK", "blocksparse_64k")
    parity.check_grad(dv[:, :, rows], dv_r, "dV", "blocksparse_64k")


# ---------------------------------------------------------------- integer work

def _lists_on_gpu(mask, N, dev, offset=0):
    """offset: bytes by which the mask's device copy is shifted off its
    allocation's alignment (the builder reads 16 bytes at a time only from a
    16-byte aligned mask)."""
    mh, nT, _ = mask.shape
    nbytes = fa.fa_blocksparse_workspace_size(1, mh, N, 64, mh)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device=dev)
    flat = torch.from_numpy(np.ascontiguousarray(mask).reshape(-1))
    buf = torch.zeros(offset + flat.numel(), dtype=torch.uint8, device=dev)
    buf[offset:] = flat.to(dev)
    md = buf[offset:]
    assert fa.fa_blocksparse_build_lists(md, mh, N, ws, nbytes) == fa.FA_OK
    status_ok()
    words = ws.view(torch.int32).cpu().numpy()
    rp = words[:mh * (nT + 1)].reshape(mh, nT + 1)
    cp = words[mh * (nT + 1):2 * mh * (nT + 1)].reshape(mh, nT + 1)
    base = 2 * mh * (nT + 1)
    ci = words[base:base + mh * nT * nT].reshape(mh, nT * nT)
    ri = words[base + mh * nT * nT:base + 2 * mh * nT * nT].reshape(mh, nT * nT)
    o0 = base + 2 * mh * nT * nT
    uo = words[o0:o0 + mh * nT].reshape(mh, nT)
    nl = words[o0 + mh * nT:o0 + mh * nT + mh]
    return rp, ci, cp, ri, uo, nl


@pytest.mark.parametrize("N,mh,density,offset", [
    (128, 1, 1.0, 0), (1000, 2, 0.3, 0), (65536, 1, None, 0), (4096, 3, 0.2, 1),
    (4096, 1, 0.5, 0), (76800, 1, 0.01, 0), (262144, 1, 0.002, 0), (20000, 2, 0.05, 3)])
def test_tile_lists_bit_exact(N, mh, density, offset):
    # one mask tile row fits a warp's 512-column access (65536), several do
    # (76800: 600 tiles, 262144: 2048), aligned and misaligned masks
    dev = device()
    nT = (N + 127) // 128
    if density is None:
        mask = W.band_random_block_mask(N, seed=2005, density=0.05)
    else:
        mask = W.random_block_mask(mh, nT, seed=N, density=density)
    rp, ci, cp, ri, uo, nl = _lists_on_gpu(mask, N, dev, offset)
    rp_o, ci_o, cp_o, ri_o = oracle.mask_lists(mask)
    assert np.array_equal(rp, rp_o) and np.array_equal(cp, cp_o)
    for h in range(mask.shape[0]):
        assert np.array_equal(ci[h, :rp[h, -1]], ci_o[h])
        assert np.array_equal(ri[h, :cp[h, -1]], ri_o[h])
        # backward order: key tiles by descending column count, ties by index;
        # long key tiles: count above twice the mean (count * nT > 2 * nnz)
        cnt = np.diff(cp_o[h])
        assert np.array_equal(uo[h], np.argsort(-cnt, kind="stable"))
        assert nl[h] == int(np.count_nonzero(cnt.astype(np.int64) * nT > 2 * int(cnt.sum())))


def _schedule(N, causal, mask, dev):
    nT = (N + 127) // 128
    heads = 1 if mask is None else mask.shape[0]
    fc = torch.full((heads, nT), -1, dtype=torch.int32, device=dev)
    bc = torch.full((heads, nT), -1, dtype=torch.int32, device=dev)
    fl = torch.full((heads, nT, nT), -1, dtype=torch.int32, device=dev)
    bl = torch.full((heads, nT, nT), -1, dtype=torch.int32, device=dev)
    md, ws, nbytes = None, None, 0
    if mask is not None:
        md = torch.from_numpy(np.ascontiguousarray(mask)).to(dev)
        nbytes = fa.fa_blocksparse_workspace_size(1, heads, N, 64, heads)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    assert fa.fa_debug_schedule(N, causal, md, heads, ws, nbytes, fc, bc, fl, bl) == fa.FA_OK
    status_ok()
    return fc.cpu().numpy(), bc.cpu().numpy(), fl.cpu().numpy(), bl.cpu().numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,mask_kind", [(1, None), (1024, None), (16384, None), (1000, "rand"),
                                         (65536, "band")])
def test_schedules_bit_exact(N, mask_kind, causal):
    dev = device()
    nT = (N + 127) // 128
    mask = None
    if mask_kind == "rand":
        mask = W.random_block_mask(2, nT, seed=11, density=0.4)
    elif mask_kind == "band":
        mask = W.band_random_block_mask(N, seed=2005, density=0.05)
    fc, bc, fl, bl = _schedule(N, causal, mask, dev)
    counts = oracle.tile_counts(N, 128, causal, mask)
    assert np.array_equal(fc, counts)  # forward: tiles holding an allowed element
    if mask is None and causal:
        assert int(fc.sum()) == nT * (nT + 1) // 2
    heads = fc.shape[0]
    if mask is not None:
        rp, ci, cp, ri = oracle.mask_lists(mask)
    for h in range(heads):
        for a in range(nT):
            if mask is None:
                fexp = list(range(a + 1)) if causal else list(range(nT))
                bexp = list(range(a, nT)) if causal else list(range(nT))
            else:
                fexp = [int(x) for x in ci[h][rp[h, a]:rp[h, a + 1]] if not causal or x <= a]
                bexp = [int(x) for x in ri[h][cp[h, a]:cp[h, a + 1]] if not causal or x >= a]
            assert fl[h, a, :fc[h, a]].tolist() == fexp
            assert bc[h, a] == len(bexp) and bl[h, a, :bc[h, a]].tolist() == bexp


@pytest.mark.parametrize("causal,per_head", [(False, False), (True, False), (False, True)])
def test_blocksparse_backward_dynamic_units(causal, per_head):
    # Units are handed out at run time, long key tiles first: two kept
    # columns of every query tile, empty columns, a random 10 %, 256 units
    # on the 152 SMs; with per-head masks the heads have different long
    # columns and counts (the backward takes the largest count for all).
    # Every output against the oracle; two runs give the same dK, dV bit
    # for bit (a unit's sums never depend on which CTA ran it) and dQ to
    # rounding.
    dev = device()
    B, H, N, d = 2, 2, 8192, 64
    nT = N // 128
    mask = W.random_block_mask(H if per_head else 1, nT, seed=31, density=0.10)
    mask[0, :, 0] = 1
    mask[0, :, 17] = 1
    mask[0, :, 40:44] = 0
    mask[0, 5, 40] = 1
    if per_head:
        mask[1, :, 3] = 1
        mask[1, :, 50:52] = 0
    q, k, v, do = W.make_qkv(B, H, N, d, seed=4242 + causal)
    scale = 1.0 / d ** 0.5
    a = run_sparse(q, k, v, do, scale, causal, mask, dev)
    b = run_sparse(q, k, v, do, scale, causal, mask, dev)
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4]), "dK/dV differ between runs"
    assert (a[2].float() - b[2].float()).abs().max().item() <= \
        1e-2 * a[2].float().abs().max().item(), "dQ drifted between runs"
    o, lse, dq, dk, dv = a
    rows = parity.check_rows(N, seed=7)
    what = f"dynamic units causal={causal}"
    o_ref, lse_ref = parity.oracle_forward(q, k, v, scale, causal, mask=mask, rows=rows)
    parity.check_forward(o[:, :, rows], lse[:, :, rows], o_ref, lse_ref, what)
    dq_r, dk_r, dv_r = parity.oracle_backward(q, k, v, do, scale, causal, mask=mask, qrows=rows,
                                              krows=rows)
    parity.check_grad(dq[:, :, rows], dq_r, "dQ", what)
    parity.check_grad(dk[:, :, rows], dk_r, "dK", what)
    parity.check_grad(dv[:, :, rows], dv_r, "dV", what)
