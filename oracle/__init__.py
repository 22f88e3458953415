"""fp64 CPU oracle of exact scaled-dot-product attention.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``io_aware_exact_15_gb300``) never touches it, and the two share no code.

The arithmetic lives in ``fa_oracle.c`` (plain C, fp64, row by row); this
module only builds it with gcc, loads it with ctypes and converts arrays.
Every function states the definition it evaluates; see the C file for the
citations ("Standard Attention Implementation", "Tiling", "Recomputation"
and "Block-sparse FlashAttention" of the FlashAttention hackmd summary).

Parity status of each function (what pins it, tests/test_oracle_pins.py):
  forward          pinned: rows of P sum to one, Q=0 prefix/blocked means,
                   causal row 0, dominant key, N=1, closed-form golden cases,
                   permutation equivariance, float64 autograd cross-check
  backward         pinned: central finite differences of forward, column-sum
                   invariants, N=1, golden closed-form gradients
  grouped K/V      pinned: equals the pinned per-head path on repeated K/V,
                   group sums of its key gradients, finite differences through
                   a shared key/value row
  dropout          pinned: Philox4x32-10 known-answer vectors (through the
                   per-element byte mapping), keep-rate statistics, p = 0 is
                   exactly the undropped oracle, a closed-form two-key case,
                   finite differences of the dropped forward, and the mean
                   over seeds converging to the undropped output
  mask_lists       pinned: hand-derived golden lists, CSR/CSC transposition
  tile_counts      pinned: closed forms n(n+1)/2 and n^2, nnz of the mask
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

TILE = 128


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into liboracle.so (gcc, fp64, no fast-math)."""
    with _lock:
        fresh = os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)
        if force or not fresh:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                   "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
            subprocess.check_call(cmd)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = ctypes.POINTER(ctypes.c_long)
        ip = ctypes.POINTER(ctypes.c_int)
        u8p = ctypes.POINTER(ctypes.c_ubyte)
        L, I, D = ctypes.c_long, ctypes.c_int, ctypes.c_double
        F, U64, U32 = ctypes.c_float, ctypes.c_uint64, ctypes.c_uint32
        u32p = ctypes.POINTER(ctypes.c_uint32)
        lib.fao_forward.argtypes = [dp, dp, dp, L, L, L, L, L, D, I, u8p, L, L, lp, L, dp, dp,
                                    F, U64, U32, L, I]
        lib.fao_forward.restype = I
        lib.fao_backward.argtypes = [dp, dp, dp, dp, L, L, L, L, L, D, I, u8p, L, L, lp, L, lp,
                                     L, dp, dp, dp, F, U64, U32, L, I]
        lib.fao_backward.restype = I
        lib.fao_philox4x32_10.argtypes = [u32p, u32p, u32p]
        lib.fao_philox4x32_10.restype = None
        lib.fao_dropout_bytes.argtypes = [U64, U32, U64, U64, U64, L, u8p]
        lib.fao_dropout_bytes.restype = None
        lib.fao_mask_lists.argtypes = [u8p, L, L, ip, ip, ip, ip]
        lib.fao_mask_lists.restype = I
        lib.fao_tile_counts.argtypes = [L, L, I, u8p, L, lp]
        lib.fao_tile_counts.restype = I
        _lib = lib
    return _lib


def _threads(nthreads):
    if nthreads is None:
        return os.cpu_count() or 1
    return int(nthreads)


def _f64(a):
    a = np.asarray(a, dtype=np.float64)
    if a.ndim != 4:
        raise ValueError("expected a [B, H, N, d] array")
    return np.ascontiguousarray(a)


def _ptr(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


def _mask_args(block_mask, H):
    if block_mask is None:
        return None, 1, None
    m = np.ascontiguousarray(np.asarray(block_mask, dtype=np.uint8))
    if m.ndim == 2:
        m = m[None]
    if m.shape[0] not in (1, H) or m.shape[1] != m.shape[2]:
        raise ValueError("block mask must be [1 or H, nT, nT]")
    return m, m.shape[0], m


def _rows(rows):
    if rows is None:
        return None, 0, None
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return _ptr(r, ctypes.c_long), len(r), r


def _drop_args(dropout, batch0=0):
    """(p, seed, offset, batch0) for the C calls; dropout = None or
    (p, seed, offset) with p in [0, 1) taken in float32."""
    if dropout is None:
        return 0.0, 0, 0, 0
    p, seed, offset = dropout
    return float(np.float32(p)), int(seed), int(offset), int(batch0)


def philox4x32_10(counter, key):
    """Philox4x32-10 of a 4-word counter and a 2-word key (uint32 each)."""
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32).reshape(4))
    k_ = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    _load().fao_philox4x32_10(_ptr(c, ctypes.c_uint32), _ptr(k_, ctypes.c_uint32),
                              _ptr(out, ctypes.c_uint32))
    return out


def dropout_bytes(seed, offset, bhc, i, j0, count):
    """Random bytes of dropout elements (bhc, i, j0 .. j0+count-1), where
    bhc = b * H + h; element (i, j) is kept iff its byte >= rint(256 p)."""
    out = np.zeros(int(count), dtype=np.uint8)
    _load().fao_dropout_bytes(int(seed), int(offset), int(bhc), int(i), int(j0), int(count),
                              _ptr(out, ctypes.c_ubyte))
    return out


def dropout_threshold(p):
    """t = rint(256 p), p taken in float32: kept iff byte >= t."""
    return int(np.rint(256.0 * float(np.float32(p))))


def dropout_keep(seed, offset, p, B, H, N, batch0=0):
    """Keep indicator z [B, H, N, N] (uint8) of the dropout definition."""
    t = dropout_threshold(p)
    z = np.zeros((B, H, N, N), dtype=np.uint8)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                z[b, h, i] = dropout_bytes(seed, offset, (batch0 + b) * H + h, i, 0, N) >= t
    return z


def forward(q, k, v, scale, causal=False, block_mask=None, tile=TILE, rows=None, nthreads=None,
            dropout=None, batch0=0):
    """O and natural-log lse of softmax(scale*QK^T + mask) V in fp64.

    q: [B, H, N, d]; k, v: [B, Hkv, N, d] with H a multiple of Hkv (query
    head h reads key/value head h // (H // Hkv)).  block_mask: [1 or H, nT,
    nT] (nonzero keeps the tile), nT = ceil(N / tile).  rows: optional query
    rows evaluated in every head.  dropout: None or (p, seed, offset):
    inverted dropout of P with the Philox keep rule of fa_oracle.c (batch b
    enters the counter as batch0 + b).  Returns o [B, H, R, d] and lse
    [B, H, R] (R = N or len(rows)).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    m, mh, keep = _mask_args(block_mask, H)
    rp, nr, keep_r = _rows(rows)
    R = N if rows is None else nr
    o = np.zeros((B, H, R, d))
    lse = np.zeros((B, H, R))
    st = _load().fao_forward(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                             _ptr(v, ctypes.c_double), B, H, Hkv, N, d, float(scale),
                             int(bool(causal)),
                             None if m is None else _ptr(m, ctypes.c_ubyte), mh, tile, rp, nr,
                             _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                             *_drop_args(dropout, batch0), _threads(nthreads))
    if st != 0:
        raise ValueError(f"oracle forward rejected its arguments ({st})")
    return o, lse


def backward(q, k, v, do, scale, causal=False, block_mask=None, tile=TILE, qrows=None,
             krows=None, nthreads=None, dropout=None, batch0=0):
    """dQ, dK, dV of sum(O * dO) for O = softmax(scale*QK^T + mask) V, fp64.

    qrows / krows: optional query / key rows evaluated in every head.  With
    k, v of Hkv < H heads, dk and dv sum over the query heads of each group.
    dropout, batch0: as forward.  Returns dq [B,H,Rq,d], dk [B,Hkv,Rk,d], dv [B,Hkv,Rk,d].
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    m, mh, keep = _mask_args(block_mask, H)
    qp, nq, keep_q = _rows(qrows)
    kp, nk, keep_k = _rows(krows)
    Rq = N if qrows is None else nq
    Rk = N if krows is None else nk
    dq = np.zeros((B, H, Rq, d))
    dk = np.zeros((B, Hkv, Rk, d))
    dv = np.zeros((B, Hkv, Rk, d))
    st = _load().fao_backward(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                              _ptr(v, ctypes.c_double), _ptr(do, ctypes.c_double), B, H, Hkv, N, d,
                              float(scale), int(bool(causal)),
                              None if m is None else _ptr(m, ctypes.c_ubyte), mh, tile, qp, nq, kp,
                              nk, _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double),
                              _ptr(dv, ctypes.c_double), *_drop_args(dropout, batch0),
                              _threads(nthreads))
    if st != 0:
        raise ValueError(f"oracle backward failed ({st})")
    return dq, dk, dv


def mask_lists(block_mask):
    """CSR (per query tile, ascending key tiles) and CSC (per key tile,
    ascending query tiles) of a [Hm, nT, nT] block mask.

    Returns (row_ptr [Hm, nT+1], col_idx list of Hm arrays, col_ptr, row_idx).
    """
    m = np.ascontiguousarray(np.asarray(block_mask, dtype=np.uint8))
    if m.ndim == 2:
        m = m[None]
    Hm, nT, _ = m.shape
    rp = np.zeros((Hm, nT + 1), dtype=np.int32)
    cp = np.zeros((Hm, nT + 1), dtype=np.int32)
    ci = np.zeros((Hm, nT * nT), dtype=np.int32)
    ri = np.zeros((Hm, nT * nT), dtype=np.int32)
    st = _load().fao_mask_lists(_ptr(m, ctypes.c_ubyte), Hm, nT, _ptr(rp, ctypes.c_int),
                                _ptr(ci, ctypes.c_int), _ptr(cp, ctypes.c_int),
                                _ptr(ri, ctypes.c_int))
    if st != 0:
        raise ValueError("oracle mask_lists rejected its arguments")
    return rp, [ci[h, :rp[h, -1]].copy() for h in range(Hm)], cp, \
        [ri[h, :cp[h, -1]].copy() for h in range(Hm)]


def tile_counts(N, tile=TILE, causal=False, block_mask=None):
    """Per query tile: how many key tiles hold an allowed element (brute force)."""
    nT = (N + tile - 1) // tile
    if block_mask is None:
        m, mh = None, 1
    else:
        m = np.ascontiguousarray(np.asarray(block_mask, dtype=np.uint8))
        if m.ndim == 2:
            m = m[None]
        mh = m.shape[0]
    out = np.zeros((mh, nT), dtype=np.int64)
    st = _load().fao_tile_counts(N, tile, int(bool(causal)),
                                 None if m is None else _ptr(m, ctypes.c_ubyte), mh,
                                 _ptr(out, ctypes.c_long))
    if st != 0:
        raise ValueError("oracle tile_counts rejected its arguments")
    return out


# ------------------------------------------------------------------ variable-length batches
def _seq_bounds(cu_seqlens):
    cu = [int(x) for x in np.asarray(cu_seqlens).reshape(-1)]
    if len(cu) < 2 or cu[0] != 0 or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must start at 0 and be non-decreasing")
    return cu


def forward_varlen(q, k, v, cu_seqlens, scale, causal=False, nthreads=None, dropout=None):
    """Packed variable-length batch: q, k, v are [H, T, d] with sequence b
    in tokens cu_seqlens[b] .. cu_seqlens[b+1]; attention stays inside each
    sequence (the padding-mask benchmark of the summary's section 4.4).
    Evaluates the per-sequence definition above; with dropout, sequence b
    is batch b of the dropout counter.  Returns o [H, T, d] and lse [H, T]."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    cu = _seq_bounds(cu_seqlens)
    H, T, d = q.shape
    o = np.zeros((H, T, d))
    lse = np.full((H, T), -np.inf)
    for s, (a, b) in enumerate(zip(cu, cu[1:])):
        if b == a:
            continue
        ob, lb = forward(q[None, :, a:b], k[None, :, a:b], v[None, :, a:b], scale, causal=causal,
                         nthreads=nthreads, dropout=dropout, batch0=s)
        o[:, a:b] = ob[0]
        lse[:, a:b] = lb[0]
    return o, lse


def backward_varlen(q, k, v, do, cu_seqlens, scale, causal=False, nthreads=None, dropout=None):
    """Gradients of sum(O * dO) for forward_varlen; each [H, T, d]."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    cu = _seq_bounds(cu_seqlens)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for s, (a, b) in enumerate(zip(cu, cu[1:])):
        if b == a:
            continue
        g = backward(q[None, :, a:b], k[None, :, a:b], v[None, :, a:b], do[None, :, a:b], scale,
                     causal=causal, nthreads=nthreads, dropout=dropout, batch0=s)
        dq[:, a:b], dk[:, a:b], dv[:, a:b] = g[0][0], g[1][0], g[2][0]
    return dq, dk, dv
