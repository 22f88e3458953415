"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test targets a different way the oracle could be wrong (a dropped
term, a wrong sign or index, a transposed operand, a mask off by one), and
none of them re-evaluates the oracle's own formula:

* hand-derived closed-form cases (tests/golden), forward and gradients;
* rows of P sum to one (V = 1 gives O = 1);
* Q = 0 gives uniform weights: the (causal / block-masked) mean of V rows
  and lse = ln(number of allowed keys);
* causal row 0 attends only to key 0; N = 1;
* a dominant key returns its value row;
* permutation equivariance;
* central finite differences of the forward pin the backward;
* column-sum invariants of the gradients;
* integer work: hand-derived lists, transposition, closed-form tile counts.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _as4(x):
    return np.asarray(x, dtype=np.float64)[None, None]


# --------------------------------------------------------------------------
# golden closed-form cases

@pytest.mark.parametrize("variant", ["dense", "causal"])
def test_golden_two_keys(golden_dir, variant):
    g = _golden(golden_dir, "closed_form_two_keys.json")
    q, k, v, do = (_as4(g[n]) for n in ("q", "k", "v", "dO"))
    causal = variant == "causal"
    o, lse = oracle.forward(q, k, v, g["scale"], causal=causal)
    exp = g[variant]
    np.testing.assert_allclose(o[0, 0], exp["o"], atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], exp["lse"], atol=1e-14)
    dq, dk, dv = oracle.backward(q, k, v, do, g["scale"], causal=causal)
    np.testing.assert_allclose(dq[0, 0], exp["dq"], atol=1e-14)
    np.testing.assert_allclose(dk[0, 0], exp["dk"], atol=1e-14)
    np.testing.assert_allclose(dv[0, 0], exp["dv"], atol=1e-14)


def test_golden_element_mask(golden_dir):
    g = _golden(golden_dir, "closed_form_element_mask.json")
    q, k, v, do = (_as4(g[n]) for n in ("q", "k", "v", "dO"))
    mask = np.asarray(g["mask"], dtype=np.uint8)[None]
    o, lse = oracle.forward(q, k, v, g["scale"], block_mask=mask, tile=g["tile"])
    np.testing.assert_allclose(o[0, 0], g["o"], atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], g["lse"], atol=1e-14)
    dq, dk, dv = oracle.backward(q, k, v, do, g["scale"], block_mask=mask, tile=g["tile"])
    np.testing.assert_allclose(dq[0, 0], g["dq"], atol=1e-14)
    np.testing.assert_allclose(dk[0, 0], g["dk"], atol=1e-14)
    np.testing.assert_allclose(dv[0, 0], g["dv"], atol=1e-14)


# --------------------------------------------------------------------------
# forward invariants and special cases

@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(causal):
    rng = np.random.default_rng(0)
    B, H, N, d = 2, 3, 37, 8
    q, k = _rand(rng, B, H, N, d), _rand(rng, B, H, N, d)
    v = np.ones((B, H, N, d))
    o, _ = oracle.forward(q, k, v, 0.7, causal=causal)
    np.testing.assert_allclose(o, 1.0, atol=1e-12)


def test_rows_of_p_sum_to_one_blocksparse():
    rng = np.random.default_rng(1)
    B, H, N, d, T = 1, 2, 40, 4, 8
    nT = N // T
    mask = (rng.random((H, nT, nT)) < 0.5).astype(np.uint8)
    mask[:, :, 0] = 1
    q, k = _rand(rng, B, H, N, d), _rand(rng, B, H, N, d)
    o, _ = oracle.forward(q, k, np.ones((B, H, N, d)), 1.3, block_mask=mask, tile=T)
    np.testing.assert_allclose(o, 1.0, atol=1e-12)


def test_zero_query_dense_causal_and_blocked_means():
    rng = np.random.default_rng(2)
    B, H, N, d, T = 1, 2, 24, 5, 6
    q = np.zeros((B, H, N, d))
    k, v = _rand(rng, B, H, N, d), _rand(rng, B, H, N, d)
    o, lse = oracle.forward(q, k, v, 0.5)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape),
                               atol=1e-13)
    np.testing.assert_allclose(lse, math.log(N), atol=1e-13)
    o, lse = oracle.forward(q, k, v, 0.5, causal=True)
    prefix = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    np.testing.assert_allclose(o, prefix, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], np.log(np.arange(1, N + 1)), atol=1e-13)
    nT = N // T
    mask = (rng.random((H, nT, nT)) < 0.5).astype(np.uint8)
    mask[:, 1, :] = 0  # an empty row of tiles
    o, lse = oracle.forward(q, k, v, 0.5, block_mask=mask, tile=T)
    for h in range(H):
        for i in range(N):
            keys = [j for j in range(N) if mask[h, i // T, j // T]]
            if not keys:
                np.testing.assert_array_equal(o[0, h, i], 0.0)
                assert lse[0, h, i] == -np.inf
            else:
                np.testing.assert_allclose(o[0, h, i], v[0, h, keys].mean(axis=0), atol=1e-13)
                np.testing.assert_allclose(lse[0, h, i], math.log(len(keys)), atol=1e-13)


def test_causal_row0_and_single_key():
    rng = np.random.default_rng(3)
    B, H, N, d = 2, 2, 9, 6
    q, k, v = (_rand(rng, B, H, N, d) for _ in range(3))
    o, lse = oracle.forward(q, k, v, 0.3, causal=True)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0], 0.3 * np.sum(q[:, :, 0] * k[:, :, 0], axis=-1),
                               atol=1e-13)


def test_n_equals_one():
    rng = np.random.default_rng(4)
    q, k, v, do = (_rand(rng, 2, 3, 1, 7) for _ in range(4))
    o, lse = oracle.forward(q, k, v, 0.9)
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse[..., 0], 0.9 * np.sum(q[..., 0, :] * k[..., 0, :], -1),
                               atol=1e-14)
    dq, dk, dv = oracle.backward(q, k, v, do, 0.9)
    np.testing.assert_allclose(dv, do, atol=1e-15)
    np.testing.assert_allclose(dq, 0.0, atol=1e-15)
    np.testing.assert_allclose(dk, 0.0, atol=1e-15)


def test_dominant_key_returns_its_value():
    rng = np.random.default_rng(5)
    N, d = 16, 8
    q, k, v = (_rand(rng, 1, 1, N, d) for _ in range(3))
    i, jstar = 5, 11
    k[0, 0, jstar] = 40.0 * q[0, 0, i] / np.linalg.norm(q[0, 0, i])
    o, _ = oracle.forward(q, k, v, 1.0)
    # gap between the dominant score and the others exceeds 30 here
    s = k[0, 0] @ q[0, 0, i]
    gap = s[jstar] - np.max(np.delete(s, jstar))
    assert gap > 20
    np.testing.assert_allclose(o[0, 0, i], v[0, 0, jstar], atol=N * math.exp(-gap) * 10)


def test_permutation_equivariance():
    rng = np.random.default_rng(6)
    B, H, N, d = 1, 2, 21, 5
    q, k, v = (_rand(rng, B, H, N, d) for _ in range(3))
    o, lse = oracle.forward(q, k, v, 0.8)
    pk = rng.permutation(N)
    o2, lse2 = oracle.forward(q, k[:, :, pk], v[:, :, pk], 0.8)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, atol=1e-13)
    pq = rng.permutation(N)
    o3, lse3 = oracle.forward(q[:, :, pq], k, v, 0.8)
    np.testing.assert_allclose(o3, o[:, :, pq], atol=1e-13)
    np.testing.assert_allclose(lse3, lse[:, :, pq], atol=1e-13)


def test_lse_is_log_of_plain_exp_sum():
    rng = np.random.default_rng(7)
    N, d = 12, 4
    q, k, v = (_rand(rng, 1, 1, N, d) for _ in range(3))
    _, lse = oracle.forward(q, k, v, 0.5)
    for i in range(N):
        direct = math.log(math.fsum(math.exp(0.5 * float(np.dot(q[0, 0, i], k[0, 0, j])))
                                    for j in range(N)))
        assert abs(lse[0, 0, i] - direct) < 1e-13


def test_row_subset_matches_full():
    rng = np.random.default_rng(8)
    B, H, N, d = 1, 3, 50, 4
    q, k, v, do = (_rand(rng, B, H, N, d) for _ in range(4))
    rows = np.array([0, 7, 8, 49])
    o, lse = oracle.forward(q, k, v, 0.6, causal=True)
    o_r, lse_r = oracle.forward(q, k, v, 0.6, causal=True, rows=rows)
    np.testing.assert_array_equal(o_r, o[:, :, rows])
    np.testing.assert_array_equal(lse_r, lse[:, :, rows])
    dq, dk, dv = oracle.backward(q, k, v, do, 0.6, causal=True)
    dq_r, dk_r, dv_r = oracle.backward(q, k, v, do, 0.6, causal=True, qrows=rows, krows=rows[::-1])
    np.testing.assert_allclose(dq_r, dq[:, :, rows], atol=1e-14)
    np.testing.assert_allclose(dk_r, dk[:, :, rows[::-1]], atol=1e-14)
    np.testing.assert_allclose(dv_r, dv[:, :, rows[::-1]], atol=1e-14)


# --------------------------------------------------------------------------
# gradients

def _loss(q, k, v, do, scale, causal, mask, tile):
    o, _ = oracle.forward(q, k, v, scale, causal=causal, block_mask=mask, tile=tile, nthreads=1)
    return float(np.sum(o * do))


@pytest.mark.parametrize("case", ["dense", "causal", "blocksparse", "blocksparse_causal"])
def test_gradients_match_central_differences(case):
    rng = np.random.default_rng(9)
    B, H, N, d, T = 1, 2, 12, 4, 4
    q, k, v, do = (_rand(rng, B, H, N, d) for _ in range(4))
    causal = "causal" in case
    mask = None
    if "blocksparse" in case:
        mask = (rng.random((H, N // T, N // T)) < 0.6).astype(np.uint8)
        mask[0, 1, :] = 0
    scale = 0.7
    dq, dk, dv = oracle.backward(q, k, v, do, scale, causal=causal, block_mask=mask, tile=T,
                                 nthreads=1)
    h = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, do, scale, causal, mask, T)
            x[idx] = old - h
            lm = _loss(q, k, v, do, scale, causal, mask, T)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(fd - g)) / max(1.0, np.max(np.abs(g)))
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_column_sums(causal):
    rng = np.random.default_rng(10)
    B, H, N, d = 2, 2, 33, 6
    q, k, v, do = (_rand(rng, B, H, N, d) for _ in range(4))
    dq, dk, dv = oracle.backward(q, k, v, do, 0.4, causal=causal)
    # sum_j dS_ij = 0 for every row  =>  sum_j dK_j = 0
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    # sum_j P_ij = 1 for every row  =>  sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)


def test_scale_folding():
    # (scale, Q) and (scale/a, a*Q) define the same scores
    rng = np.random.default_rng(11)
    q, k, v = (_rand(rng, 1, 2, 19, 4) for _ in range(3))
    o1, l1 = oracle.forward(q, k, v, 0.5, causal=True)
    o2, l2 = oracle.forward(q * 4.0, k, v, 0.125, causal=True)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_autograd_crosscheck_float64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    B, H, N, d, T = 1, 2, 48, 8, 16
    q, k, v, do = (_rand(rng, B, H, N, d) for _ in range(4))
    nT = N // T
    mask = (rng.random((1, nT, nT)) < 0.5).astype(np.uint8)
    mask[:, :, 0] = 1
    for causal, m in ((False, None), (True, None), (False, mask), (True, mask)):
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        s = 0.35 * tq @ tk.transpose(-1, -2)
        allow = torch.ones(N, N, dtype=torch.bool)
        if causal:
            allow &= torch.tril(torch.ones(N, N, dtype=torch.bool))
        if m is not None:
            allow &= torch.tensor(m[0]).bool().repeat_interleave(T, 0).repeat_interleave(T, 1)
        s = s.masked_fill(~allow, float("-inf"))
        o = torch.softmax(s, dim=-1) @ tv
        lse = torch.logsumexp(s, dim=-1)
        (o * torch.tensor(do)).sum().backward()
        oo, ll = oracle.forward(q, k, v, 0.35, causal=causal, block_mask=m, tile=T)
        dq, dk, dv = oracle.backward(q, k, v, do, 0.35, causal=causal, block_mask=m, tile=T)
        np.testing.assert_allclose(oo, o.detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(ll, lse.detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


# --------------------------------------------------------------------------
# integer work

def test_mask_lists_golden(golden_dir):
    g = _golden(golden_dir, "mask_lists_4x4.json")
    rp, ci, cp, ri = oracle.mask_lists(np.asarray(g["mask"], dtype=np.uint8))
    assert rp[0].tolist() == g["row_ptr"]
    assert ci[0].tolist() == g["col_idx"]
    assert cp[0].tolist() == g["col_ptr"]
    assert ri[0].tolist() == g["row_idx"]
    m = np.asarray(g["mask"], dtype=np.uint8)
    assert oracle.tile_counts(512, 128, False, m)[0].tolist() == g["tile_counts_dense"]
    assert oracle.tile_counts(512, 128, True, m)[0].tolist() == g["tile_counts_causal"]


def test_mask_lists_are_transposes():
    rng = np.random.default_rng(13)
    mask = (rng.random((3, 17, 17)) < 0.3).astype(np.uint8)
    rp, ci, cp, ri = oracle.mask_lists(mask)
    for h in range(3):
        pairs_csr = {(a, int(b)) for a in range(17) for b in ci[h][rp[h, a]:rp[h, a + 1]]}
        pairs_csc = {(int(a), b) for b in range(17) for a in ri[h][cp[h, b]:cp[h, b + 1]]}
        assert pairs_csr == pairs_csc
        assert len(pairs_csr) == int(mask[h].sum()) == rp[h, -1] == cp[h, -1]
        for a in range(17):
            seg = ci[h][rp[h, a]:rp[h, a + 1]]
            assert np.all(np.diff(seg) > 0)


@pytest.mark.parametrize("N", [1, 127, 128, 129, 1000, 1024])
def test_tile_counts_closed_forms(N):
    n = (N + 127) // 128
    dense = oracle.tile_counts(N, 128, False)
    causal = oracle.tile_counts(N, 128, True)
    assert dense[0].tolist() == [n] * n
    assert causal[0].tolist() == list(range(1, n + 1))
    assert int(causal.sum()) == n * (n + 1) // 2


# --------------------------------------------------------------------------
# grouped key/value heads (H query heads share Hkv key/value heads)

@pytest.mark.parametrize("causal", [False, True])
def test_grouped_kv_equals_repeated_kv(causal):
    rng = np.random.default_rng(14)
    B, H, Hkv, N, d = 2, 6, 2, 19, 5
    G = H // Hkv
    q, do = _rand(rng, B, H, N, d), _rand(rng, B, H, N, d)
    k, v = _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    o, lse = oracle.forward(q, k, v, 0.45, causal=causal)
    o_r, lse_r = oracle.forward(q, kr, vr, 0.45, causal=causal)
    np.testing.assert_allclose(o, o_r, atol=1e-14)
    np.testing.assert_allclose(lse, lse_r, atol=1e-14)
    dq, dk, dv = oracle.backward(q, k, v, do, 0.45, causal=causal)
    dq_r, dk_r, dv_r = oracle.backward(q, kr, vr, do, 0.45, causal=causal)
    np.testing.assert_allclose(dq, dq_r, atol=1e-13)
    # a shared parameter's gradient is the sum over its uses
    np.testing.assert_allclose(dk, dk_r.reshape(B, Hkv, G, N, d).sum(axis=2), atol=1e-13)
    np.testing.assert_allclose(dv, dv_r.reshape(B, Hkv, G, N, d).sum(axis=2), atol=1e-13)


def test_grouped_kv_gradients_match_central_differences():
    rng = np.random.default_rng(15)
    B, H, Hkv, N, d = 1, 4, 1, 9, 3
    q, do = _rand(rng, B, H, N, d), _rand(rng, B, H, N, d)
    k, v = _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
    dq, dk, dv = oracle.backward(q, k, v, do, 0.6, causal=True, nthreads=1)
    h = 1e-5

    def loss():
        o, _ = oracle.forward(q, k, v, 0.6, causal=True, nthreads=1)
        return float(np.sum(o * do))

    for x, g in ((k, dk), (v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = loss()
            x[idx] = old - h
            lm = loss()
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        assert np.max(np.abs(fd - g)) / max(1.0, np.max(np.abs(g))) < 1e-6


def test_grouped_kv_rejects_bad_groups():
    rng = np.random.default_rng(16)
    q, k = _rand(rng, 1, 4, 8, 2), _rand(rng, 1, 3, 8, 2)
    with pytest.raises(ValueError):
        oracle.forward(q, k, k, 1.0)


# --------------------------------------------------------------------------
# variable-length batches: the block-diagonal mask of packed sequences

def _block_diag_mask(cu, causal):
    T = cu[-1]
    m = np.zeros((1, T, T), dtype=np.uint8)
    for a, b in zip(cu, cu[1:]):
        m[0, a:b, a:b] = 1
    if causal:
        m[0] &= np.tril(np.ones((T, T), dtype=np.uint8))
    return m


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_packed_block_diagonal_mask(causal):
    rng = np.random.default_rng(17)
    cu = [0, 5, 5, 12, 30]  # includes an empty sequence
    H, T, d = 2, cu[-1], 4
    q, k, v, do = (_rand(rng, H, T, d) for _ in range(4))
    o, lse = oracle.forward_varlen(q, k, v, cu, 0.55, causal=causal)
    dq, dk, dv = oracle.backward_varlen(q, k, v, do, cu, 0.55, causal=causal)
    # same problem as one packed sequence with an element mask (tile 1): a
    # different path through the oracle
    m = _block_diag_mask(cu, causal)
    o2, lse2 = oracle.forward(q[None], k[None], v[None], 0.55, block_mask=m, tile=1)
    g2 = oracle.backward(q[None], k[None], v[None], do[None], 0.55, block_mask=m, tile=1)
    np.testing.assert_allclose(o, o2[0], atol=1e-13)
    np.testing.assert_allclose(lse, lse2[0], atol=1e-13)
    for a, b in ((dq, g2[0]), (dk, g2[1]), (dv, g2[2])):
        np.testing.assert_allclose(a, b[0], atol=1e-12)


def test_varlen_equal_lengths_equals_batch():
    rng = np.random.default_rng(18)
    B, H, N, d = 3, 2, 11, 4
    q, k, v = (_rand(rng, B, H, N, d) for _ in range(3))
    pack = lambda x: np.concatenate([x[b] for b in range(B)], axis=1)  # [H, B*N, d]
    o, lse = oracle.forward_varlen(pack(q), pack(k), pack(v), [0, 11, 22, 33], 0.3, causal=True)
    o_b, lse_b = oracle.forward(q, k, v, 0.3, causal=True)
    np.testing.assert_allclose(o, pack(o_b), atol=1e-14)
    np.testing.assert_allclose(lse, np.concatenate([lse_b[b] for b in range(B)], axis=1),
                               atol=1e-14)
