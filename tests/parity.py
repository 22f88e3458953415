"""Shared helpers for the GPU parity tests: run the CUDA path through the
C ABI and the fp64 oracle on the same seeded bf16 inputs, and compare.

Tolerances (bf16 inputs, fp32 accumulation; written once here):
  O      max |diff| <= 2e-2 and mean |diff| <= 2e-3
  lse    max |diff| <= 1e-2
  dQ, dK, dV   max |diff| / max(max |ref|, 1e-3) <= 5e-2 per tensor
The 1e-3 floor only matters when the exact gradient is identically zero
(N = 1 gives dQ = dK = 0): the relative bound is then undefined and the
check becomes |diff| <= 5e-5.
"""
from __future__ import annotations

import numpy as np

import oracle

O_MAX, O_MEAN, LSE_MAX, GRAD_REL, GRAD_FLOOR = 2e-2, 2e-3, 1e-2, 5e-2, 1e-3


def f64(t):
    return t.detach().float().cpu().double().numpy()


def check_forward(o_gpu, lse_gpu, o_ref, lse_ref, what="", o_scale=1.0):
    """o_scale: the factor O's magnitude carries beyond the undropped
    output's (dropout's keep scale 1 / (1 - p')); the O bounds scale by it."""
    o = f64(o_gpu)
    lse = lse_gpu.detach().cpu().double().numpy()
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX * o_scale, f"{what}: O max err {err.max():.3e}"
    assert err.mean() <= O_MEAN * o_scale, f"{what}: O mean err {err.mean():.3e}"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
    if fin.any():
        le = np.abs(lse[fin] - lse_ref[fin]).max()
        assert le <= LSE_MAX, f"{what}: lse max err {le:.3e}"
    return float(err.max()), float(err.mean())


def check_grad(g_gpu, g_ref, name, what="", floor=GRAD_FLOOR):
    """floor: the scale below which the bound stops being relative (see
    cancel_floor for gradients that are zero by cancellation)."""
    g = f64(g_gpu) if not isinstance(g_gpu, np.ndarray) else g_gpu
    assert np.all(np.isfinite(g)), f"{what}: non-finite {name}"
    scale = max(np.abs(g_ref).max(), floor)
    rel = np.abs(g - g_ref).max() / scale
    assert rel <= GRAD_REL, f"{what}: {name} rel err {rel:.3e}"
    return float(rel)


def oracle_forward(q, k, v, scale, causal=False, mask=None, rows=None):
    return oracle.forward(f64(q), f64(k), f64(v), scale, causal=causal, block_mask=mask,
                          rows=rows)


def oracle_backward(q, k, v, do, scale, causal=False, mask=None, qrows=None, krows=None,
                    heads=None):
    """Oracle gradients; `heads` restricts the evaluation to a list of
    (b, h) pairs (returns arrays over those heads only)."""
    qa, ka, va, da = f64(q), f64(k), f64(v), f64(do)
    if heads is None:
        return oracle.backward(qa, ka, va, da, scale, causal=causal, block_mask=mask,
                               qrows=qrows, krows=krows)
    outs = []
    for (b, h) in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        m = None
        if mask is not None:
            m = mask if mask.shape[0] == 1 else mask[h:h + 1]
        outs.append(oracle.backward(qa[sl], ka[sl], va[sl], da[sl], scale, causal=causal,
                                    block_mask=m, qrows=qrows, krows=krows))
    return tuple(np.concatenate([o[i] for o in outs], axis=1) for i in range(3))


def cancel_floor(scale, o, do, other):
    """Scale of the terms that cancel in a gradient that is exactly zero
    (one key per row: dS = P (dP - D) = 0).  The kernel forms D from the
    bf16-rounded O, so the cancellation leaves |dD| <= 2^-8 sum_c |dO O|,
    and dQ (dK) moves by at most scale * |dD| * max|K| (max|Q|).  Returns
    scale * max_i sum_c |dO_ic O_ic| * max|other|."""
    o_, do_, x = f64(o), f64(do), f64(other)
    return float(scale * np.abs(do_ * o_).sum(-1).max() * np.abs(x).max())


def keep_scale(p):
    """1 / (1 - p') of dropout probability p (p' = rint(256 p) / 256)."""
    t = int(np.rint(256.0 * float(np.float32(p))))
    return 256.0 / (256 - t)


# ------------------------------------------------------------------ row and head samples
ORACLE_BUDGET = 2.0e11  # oracle flops per shape for the backward's heads


def check_rows(N, seed):
    """256 seeded rows and one seeded row in every 128-row tile (sorted,
    distinct), so that every query and key tile of a head is represented."""
    import fa_workloads as W
    rows = set(W.sample_rows(N, 256, seed).tolist())
    rng = np.random.default_rng(seed)
    for t in range((N + 127) // 128):
        lo, hi = 128 * t, min(N, 128 * t + 128)
        rows.add(int(rng.integers(lo, hi)))
    return np.array(sorted(rows), dtype=np.int64)


def last_round_heads(B, H, N, causal, sms, Hkv=None):
    """(batch, key/value head) pairs holding a unit of the persistent
    backward's last round: one CTA per SM takes units blockIdx.x,
    blockIdx.x + grid, ...; a unit is one key/value head x one key tile,
    numbered head-major (dense) or key-tile-major (causal)."""
    Hk = H if Hkv is None else Hkv
    nT = (N + 127) // 128
    BH = B * Hk
    units = BH * nT
    grid = min(units, sms)
    rounds = (units + grid - 1) // grid
    first = (rounds - 1) * grid
    bhs = sorted({(u // nT) if not causal else (u % BH) for u in range(first, units)})
    return [divmod(bh, Hk) for bh in bhs]


def backward_heads(w, sms, budget=ORACLE_BUDGET):
    """Heads on which a backward is compared with the oracle: all of them
    when their oracle cost (4 N^2 d flops per head, half when causal) fits
    `budget`, else that many: the first and last head, the first and last
    head of the backward's last round, and seeded others."""
    B, H, N, d = w.B, w.H, w.N, w.d
    per_head = 4.0 * N * N * d / (2 if w.causal else 1)
    n = int(min(B * H, max(4, budget // per_head)))
    if n >= B * H:
        return [(b, h) for b in range(B) for h in range(H)]
    last = last_round_heads(B, H, N, w.causal, sms)
    heads = []
    for x in [(0, 0), (B - 1, H - 1), last[0], last[-1]]:
        if x not in heads:
            heads.append(x)
    rng = np.random.default_rng(w.seed + N + d)
    for bh in rng.permutation(B * H):
        if len(heads) >= n:
            break
        x = divmod(int(bh), H)
        if x not in heads:
            heads.append(x)
    return sorted(heads)
